"""Seeded synthetic inputs shaped like the draft head's projection workloads.

This module only draws random numbers; it holds none of the method's
arithmetic (no quantisation, normalisation or products).  Both the tests'
oracle side and the GPU side take their inputs from here, so they see the
same bytes.

Recipe (the pages print no dataset; every input is synthetic):
  * Tensor t of workload c is drawn from its own generator seeded with
    ``16 * (c - 1) + t``; normal draws are made in FP32 and rounded to BF16
    (round-to-nearest-even) by ``.to(torch.bfloat16)``.
  * lm_head_m1   (32768 x 4096 reduced-vocab LM head, M=1 with RMSNorm):
    W ~ N(0, 0.02) with round(0.01 N) rows, picked by a seeded permutation,
    multiplied by 8; gamma = 1 + N(0, 0.05); H[1000, 4096] ~ N(0, 1); eps 1e-6.
  * propose_m8   (151936 x 5120 LM head, no norm; M in 1..8, and 16 / 32 for
    the batch-16 and batch-32 draft widths): W ~ N(0, 0.02) with every 16-element K block
    multiplied by 2^u, u ~ U[-6, 2] per block; X[m, 5120] ~ N(0, 1), m = 8
    by default (a call at batch M uses rows 0..M-1).
  * fc_combiner  (5120 x 10240 fc, two RMSNorms + concat; M in 1..8, and up
    to 32): W ~ N(0, 0.015); E, H [m, 5120] ~ N(0, 1), m = 8 by default;
    gamma_e, gamma_h = 1 + N(0, 0.05).
  * prefill_gemm (2048 x 17408 x 5120): A ~ N(0, 1); W ~ N(0, 0.02).
  * tiny         (256 x 512, M=1): W ~ N(0, 0.02); x ~ N(0, 1).
Every generator accepts smaller shapes so the same recipe serves parity
tests that the CPU oracle finishes in seconds.
"""
from dataclasses import dataclass, field
from typing import Optional

import torch

WORKLOAD_IDS = {"tiny": 1, "lm_head_m1": 2, "propose_m8": 3, "fc_combiner": 4,
                "prefill_gemm": 5}


def _gen(workload: str, t: int, device) -> torch.Generator:
    c = WORKLOAD_IDS[workload]
    g = torch.Generator(device=device)
    g.manual_seed(16 * (c - 1) + t)
    return g


def _normal(shape, std, workload, t, device, mean=0.0):
    g = _gen(workload, t, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


@dataclass
class GemvCase:
    """Inputs of one GEMV workload: BF16 weight to quantise and activations."""
    name: str
    w: torch.Tensor                      # BF16 [n, k]
    segments: list                       # [(x BF16 [m, k_seg], gamma BF16 [k_seg] or None)]
    eps: float = 1e-6
    extra: dict = field(default_factory=dict)

    @property
    def n(self):
        return self.w.shape[0]

    @property
    def k(self):
        return self.w.shape[1]


def tiny(n=256, k=512, m=1, device="cpu") -> GemvCase:
    w = _normal((n, k), 0.02, "tiny", 0, device).to(torch.bfloat16)
    x = _normal((m, k), 1.0, "tiny", 1, device).to(torch.bfloat16)
    return GemvCase("tiny", w, [(x, None)])


def lm_head_m1(n=32768, k=4096, rows=1000, device="cpu") -> GemvCase:
    w = _normal((n, k), 0.02, "lm_head_m1", 0, device)
    n_out = int(round(0.01 * n))
    perm = torch.randperm(n, generator=_gen("lm_head_m1", 1, device), device=device)
    w[perm[:n_out]] *= 8.0
    w = w.to(torch.bfloat16)
    gamma = _normal((k,), 0.05, "lm_head_m1", 2, device, mean=1.0).to(torch.bfloat16)
    h = _normal((rows, k), 1.0, "lm_head_m1", 3, device).to(torch.bfloat16)
    return GemvCase("lm_head_m1", w, [(h, gamma)], eps=1e-6,
                    extra={"outlier_rows": perm[:n_out].sort().values})


def propose_m8(n=151936, k=5120, m=8, device="cpu") -> GemvCase:
    w = _normal((n, k), 0.02, "propose_m8", 0, device)
    gu = _gen("propose_m8", 1, device)
    u = torch.rand((n, k // 16), generator=gu, device=device, dtype=torch.float32)
    u.mul_(8.0).sub_(6.0)                              # U[-6, 2]
    w.view(n, k // 16, 16).mul_(torch.exp2(u).unsqueeze(-1))
    del u
    w = w.to(torch.bfloat16)
    x = _normal((m, k), 1.0, "propose_m8", 2, device).to(torch.bfloat16)
    return GemvCase("propose_m8", w, [(x, None)])


def fc_combiner(n=5120, k_seg=5120, m=8, device="cpu") -> GemvCase:
    w = _normal((n, 2 * k_seg), 0.015, "fc_combiner", 0, device).to(torch.bfloat16)
    e = _normal((m, k_seg), 1.0, "fc_combiner", 1, device).to(torch.bfloat16)
    h = _normal((m, k_seg), 1.0, "fc_combiner", 2, device).to(torch.bfloat16)
    ge = _normal((k_seg,), 0.05, "fc_combiner", 3, device, mean=1.0).to(torch.bfloat16)
    gh = _normal((k_seg,), 0.05, "fc_combiner", 4, device, mean=1.0).to(torch.bfloat16)
    return GemvCase("fc_combiner", w, [(e, ge), (h, gh)], eps=1e-6)


@dataclass
class GemmCase:
    name: str
    a: torch.Tensor      # BF16 [m, k]
    w: torch.Tensor      # BF16 [n, k]


def prefill_gemm(m=2048, n=17408, k=5120, device="cpu") -> GemmCase:
    a = _normal((m, k), 1.0, "prefill_gemm", 0, device).to(torch.bfloat16)
    w = _normal((n, k), 0.02, "prefill_gemm", 1, device).to(torch.bfloat16)
    return GemmCase("prefill_gemm", a, w)


def bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit pattern (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def from_bits(b, device="cpu") -> torch.Tensor:
    """numpy uint16 bit pattern -> BF16 tensor."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
        torch.bfloat16).to(device)
