"""Run one library call on a named workload a few times (for profilers).

    python -m nvfp4_speculative_draft_gb300.profile_case --case propose --m 8 --iters 3

Cases (seeded synthetic inputs of the draft head's workloads, built on the
device): ``lm_head`` (32768 x 4096, RMSNorm + GEMV + argmax, M=1), ``propose``
(151936 x 5120 GEMV + argmax, M=--m), ``fc`` (5120 x 10240, two RMSNorms +
concat, BF16 out, M=--m), ``gemm`` (2048 x 17408 x 5120 prefill GEMM on BF16
operands, as the benchmark times it; ``gemm_f16`` with the FP16 staging
workspace),
``quantize`` (17408 x 5120), ``propose_fp8`` / ``quantize_fp8`` (the FP8
weight variant of the 151936 x 5120 head).  Inputs are prepared first (their kernels run
before the measured calls, so ``ncu -k regex:<kernel> -s <n>`` can skip them),
then the call runs --iters times and the process exits 0.
"""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import nvfp4_speculative_draft_gb300 as nd
    import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", required=True,
                    choices=["lm_head", "propose", "propose_fp8", "fc", "gemm", "gemm_f16", "quantize",
                             "quantize_fp8"])
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    nd.load()
    dev = torch.device("cuda:0")
    if args.case == "lm_head":
        c = workloads.lm_head_m1(rows=args.iters, device=dev)
        wq, _ = nd.nvfp4_quantize(c.w)
        h, gamma = c.segments[0]
        torch.cuda.synchronize()
        for i in range(args.iters):
            nd.w4a16_gemv_argmax([(h[i:i + 1], gamma, 1e-6)], wq, logits=False)
    elif args.case == "propose":
        c = workloads.propose_m8(m=max(8, args.m), device=dev)
        wq, _ = nd.nvfp4_quantize(c.w)
        x = c.segments[0][0][:args.m].contiguous()
        del c
        torch.cuda.synchronize()
        torch.cuda.empty_cache()  # keep only the quantised weight resident
        for _ in range(args.iters):
            nd.w4a16_gemv_argmax([(x, None)], wq)
    elif args.case in ("propose_fp8", "quantize_fp8"):
        c = workloads.propose_m8(device=dev)
        w8 = nd.fp8w_quantize(c.w)
        x = c.segments[0][0][:args.m].contiguous()
        if args.case == "propose_fp8":
            del c
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        for _ in range(args.iters):
            if args.case == "propose_fp8":
                nd.fp8w_gemv_argmax([(x, None)], w8)
            else:
                nd.fp8w_quantize(c.w, out=w8)
    elif args.case == "fc":
        c = workloads.fc_combiner(device=dev)
        wq, _ = nd.nvfp4_quantize(c.w)
        (e, ge), (h, gh) = c.segments
        e, h = e[:args.m].contiguous(), h[:args.m].contiguous()
        torch.cuda.synchronize()
        for _ in range(args.iters):
            nd.w4a16_gemv([(e, ge, 1e-6), (h, gh, 1e-6)], wq, out_dtype=torch.bfloat16)
    elif args.case in ("gemm", "gemm_f16"):
        c = workloads.prefill_gemm(device=dev)
        wq, _ = nd.nvfp4_quantize(c.w)
        ws = None
        if args.case == "gemm_f16":
            ws = torch.empty(nd.gemm_workspace_bytes(2048, 5120), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for _ in range(args.iters):
            nd.w4a16_gemm(c.a, wq, workspace=ws)
    else:
        c = workloads.prefill_gemm(m=128, device=dev)
        torch.cuda.synchronize()
        wq = None
        for _ in range(args.iters):
            wq, _ = nd.nvfp4_quantize(c.w, out=wq)
    torch.cuda.synchronize()


if __name__ == "__main__":
    main()
