"""Mutation check of the oracle's pins (CPU only).

Each mistake in tests/oracle_mutants.py is planted in a copy of the oracle's
C source (the oracle itself is untouched), the copy is built with the
oracle's own compiler flags, and tests/test_oracle.py is run against it in a
subprocess (NVFP4_ORACLE_LIB points the oracle at the copy).  Every mutant
must make the pins fail; an unmutated copy built the same way must pass
them, so a failure cannot come from the harness itself."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from oracle import LIB_OVERRIDE_ENV
from oracle import build as oracle_build
from oracle_mutants import MUTANTS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pins_pass(src_text, workdir, tag):
    c_path = os.path.join(workdir, f"{tag}.c")
    so_path = os.path.join(workdir, f"{tag}.so")
    with open(c_path, "w") as f:
        f.write(src_text)
    oracle_build.compile_source(c_path, so_path)
    env = dict(os.environ, **{LIB_OVERRIDE_ENV: so_path})
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                        "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode in (0, 1), f"{tag}: pytest could not run the pins:\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
    return r.returncode == 0


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(oracle_build.SRC) as f:
        src = f.read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"mutant '{name}': its source text must occur exactly once"
    jobs = [("control", src)] + [(f"m{i}", src.replace(old, new)) for i, (_, old, new) in enumerate(MUTANTS)]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        passed = dict(zip([t for t, _ in jobs], ex.map(lambda j: _pins_pass(j[1], str(tmp_path), j[0]), jobs)))
    assert passed["control"], "the unmutated copy must pass the pins"
    survivors = [MUTANTS[i][0] for i in range(len(MUTANTS)) if passed[f"m{i}"]]
    assert not survivors, f"mistakes no pin catches: {survivors}"


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
