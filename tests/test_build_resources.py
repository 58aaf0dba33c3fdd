"""Every kernel of the library compiles for sm_103a without register spills.

Spilled registers turn into local-memory traffic inside the hot loops (the
gather, the sort passes, the lookups), so a change that makes any kernel spill
should be seen at build time.  Runs on CPU: nvcc cross-compiles.
"""
import concurrent.futures as cf
import glob
import os
import re
import subprocess
import tempfile

import pytest

from submanifold_sparse_convolution_gb300 import build as build_mod

CSRC = os.path.join(os.path.dirname(os.path.abspath(build_mod.__file__)), "csrc")
SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
FUNC = re.compile(r"Function properties for (\S+)")


def _ptxas_report(src, out_dir):
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    cmd = [build_mod.nvcc()] + build_mod.NVCC_FLAGS + ["-Xptxas", "-v", "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"{os.path.basename(src)}:\n{r.stderr[-2000:]}"
    return r.stdout + r.stderr


def test_no_kernel_spills_registers():
    try:
        build_mod.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    assert srcs
    with tempfile.TemporaryDirectory() as d, cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        reports = dict(zip(srcs, ex.map(lambda s: _ptxas_report(s, d), srcs)))
    spilled, seen = [], 0
    for src, text in reports.items():
        func = None
        for line in text.splitlines():
            m = FUNC.search(line)
            if m:
                func = m.group(1)
            m = SPILL.search(line)
            if m:
                seen += 1
                if int(m.group(1)) or int(m.group(2)):
                    spilled.append(f"{os.path.basename(src)}: {func}: {line.strip()}")
    assert seen > 0, "no ptxas resource report was printed"
    assert not spilled, "\n".join(spilled)
