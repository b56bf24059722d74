"""Every kernel of both library builds compiles without register spills.

ptxas reports, per kernel, its stack frame and the bytes it spills to local
memory; a spill turns register traffic into memory traffic on the hot path,
so the build must show none.  Runs on CPU (nvcc cross-compiles for sm_103a).
The register counts are printed for the record (pytest -s)."""
import os
import re
import shutil
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

from kda_linear_attention_gated_gb300 import _build

ENTRY = re.compile(r"Compiling entry function '(\S+)'")
SPILL = re.compile(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads")
REGS = re.compile(r"Used (\d+) registers")


def _ptxas_report(state16: bool):
    with tempfile.TemporaryDirectory() as d:
        cmd = _build.nvcc_command(state16, os.path.join(d, "probe.so"), ["-Xptxas", "-v"])
        proc = subprocess.run(cmd, capture_output=True, text=True)
    assert proc.returncode == 0, proc.stderr[-2000:]
    kernels, name, spill = [], None, None
    for line in proc.stderr.splitlines():
        m = ENTRY.search(line)
        if m:
            name = m.group(1)
        m = SPILL.search(line)
        if m:
            spill = tuple(int(x) for x in m.groups())
        m = REGS.search(line)
        if m and name is not None:
            kernels.append((name, int(m.group(1)), spill))
            name, spill = None, None
    return kernels


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_every_kernel_compiles_without_spills():
    with ThreadPoolExecutor(2) as ex:
        reports = dict(zip((False, True), ex.map(_ptxas_report, (False, True))))
    seen = 0
    for state16, kernels in reports.items():
        assert kernels, "ptxas reported no kernels"
        for name, regs, (stack, stores, loads) in kernels:
            print(f"libkda_h{int(state16)} {regs:4d} registers  {name}")
            assert stores == 0 and loads == 0, f"{name}: {stores} B spill stores, {loads} B spill loads"
            seen += 1
    # decode, verify, conv, checkpoint and both prefill passes, in each build
    assert seen >= 2 * 6
