"""All 2^32 fp32 patterns through the oracle's three conversions, checked by
an independent value-based C program (tests/rne_exhaustive_check.c)."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import pytest

import oracle

HERE = Path(__file__).resolve().parent


@pytest.mark.slow
def test_conversions_exhaustive(tmp_path):
    so = oracle.build()
    exe = tmp_path / "rne_check"
    cc = oracle._compiler()
    subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe),
                    str(HERE / "rne_exhaustive_check.c"), str(so), f"-Wl,-rpath,{so.parent}", "-lm"],
                   check=True)
    parts = max(1, min(32, os.cpu_count() or 1))
    total = 1 << 32
    step = total // parts

    def run(k):
        first = k * step
        count = total - first if k == parts - 1 else step
        return subprocess.run([str(exe), str(first), str(count)], capture_output=True, text=True)

    with ThreadPoolExecutor(parts) as ex:
        results = list(ex.map(run, range(parts)))
    checked = 0
    for r in results:
        assert r.returncode == 0, r.stdout + r.stderr
        checked += int(r.stdout.split()[1])
    # every non-NaN pattern: 2^32 minus 2 * (2^23 - 1) NaNs
    assert checked == total - 2 * ((1 << 23) - 1)
