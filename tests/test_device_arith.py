"""Arithmetic identities the CUDA kernels rely on, checked on the CPU with
IEEE fp32 operations (the same operations the kernels issue):

- the scales RN(amax / 127), RN(amax / 448) and RN(amax / 6) of the int8,
  fp8 and fp4 outputs are computed by one multiplication and two fused
  multiply-adds (a division with one correction step);
  tests/div_const_check.c compares each with the correctly rounded quotient
  for every fp32 amax in [2^-100, 2^128);
- the LSE merge's log1p(u) on [0, 1] by the atanh series after a division
  with one correction step; tests/log1p_series_check.c compares it with
  log1p in double for every fp32 u in [0, 1]."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import pytest

import oracle

HERE = Path(__file__).resolve().parent


@pytest.mark.parametrize("divisor", [127, 448, 6])
def test_division_by_constant_is_correctly_rounded(tmp_path, divisor):
    exe = tmp_path / "div_const_check"
    subprocess.run([oracle._compiler(), "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe),
                    str(HERE / "div_const_check.c"), "-lm"], check=True)
    exps = list(range(-100, 128))
    parts = max(1, min(16, os.cpu_count() or 1))
    chunks = [exps[i::parts] for i in range(parts)]

    def run(ch):
        return [subprocess.run([str(exe), str(divisor), str(e), str(e)], capture_output=True, text=True)
                for e in ch]

    with ThreadPoolExecutor(parts) as ex:
        results = [r for rs in ex.map(run, chunks) for r in rs]
    checked = 0
    for r in results:
        assert r.returncode == 0, r.stdout + r.stderr
        checked += int(r.stdout.split()[1])
    assert checked == len(exps) << 23


def test_log1p_series_on_unit_interval(tmp_path):
    """The LSE merge's log1p(u), u in [0, 1] (tests/log1p_series_check.c runs
    the kernel's fp32 operations, with every quotient its reciprocal-based
    division can give): every fp32 u within 3 x 2^-24 relative (plus 2^-146
    absolute where the quotient is subnormal) of log1p in double."""
    exe = tmp_path / "log1p_series_check"
    subprocess.run([oracle._compiler(), "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe),
                    str(HERE / "log1p_series_check.c"), "-lm"], check=True)
    last = 0x3F800000
    parts = 32
    step = (last + 1) // parts
    ranges = [(k * step, last if k == parts - 1 else (k + 1) * step - 1) for k in range(parts)]

    def run(r):
        return subprocess.run([str(exe), hex(r[0]), hex(r[1])], capture_output=True, text=True)

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        results = list(ex.map(run, ranges))
    checked = 0
    for r in results:
        assert r.returncode == 0, r.stdout + r.stderr
        checked += int(r.stdout.split()[1])
    assert checked == last + 1
