"""Arithmetic identities the CUDA kernels rely on, checked on the CPU with
IEEE fp32 operations (the same operations the kernels issue):

- the group scale RN(amax / 448) of the per-group fp8 output is computed by
  one multiplication and two fused multiply-adds (a division with one
  correction step); tests/div448_check.c compares it with the correctly
  rounded quotient for every fp32 amax in [2^-100, 2^128)."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import oracle

HERE = Path(__file__).resolve().parent


def test_div448_correction_step_is_correctly_rounded(tmp_path):
    exe = tmp_path / "div448_check"
    subprocess.run([oracle._compiler(), "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe),
                    str(HERE / "div448_check.c"), "-lm"], check=True)
    exps = list(range(-100, 128))
    parts = max(1, min(16, os.cpu_count() or 1))
    chunks = [exps[i::parts] for i in range(parts)]

    def run(ch):
        return [subprocess.run([str(exe), str(e), str(e)], capture_output=True, text=True) for e in ch]

    with ThreadPoolExecutor(parts) as ex:
        results = [r for rs in ex.map(run, chunks) for r in rs]
    checked = 0
    for r in results:
        assert r.returncode == 0, r.stdout + r.stderr
        checked += int(r.stdout.split()[1])
    assert checked == len(exps) << 23
