"""The linear kernels keep every value in registers: no instantiation of the
tcgen05 or mma.sync kernel, at any width, may spill to local memory.

The tcgen05 kernel runs 1024 threads at 64 registers in its 16-row-slot
class, right at the cap. A change anywhere in the kernel, even in a role off
the hot path, can push the whole kernel's allocation over it. Once, 72 bytes of
spills from a counter loop in the epilogue warps slowed the LM head's step
by 4 %. The test compiles each width's translation unit for sm_103a with the
assembler's resource report (`-Xptxas -v`, as the build does) and reads the
spill counts it prints. It needs nvcc, not a GPU.
"""

import os
import re
import shutil
import subprocess

import pytest

from trellis_quantized_linear_rot_gb300 import build as b

WIDTHS = (2, 3, 4, 5, 6, 8)


def _nvcc():
    try:
        return b.nvcc()
    except RuntimeError:
        return None


@pytest.fixture(scope="module")
def reports(tmp_path_factory):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("ptxas")
    procs = {}
    for w in WIDTHS:
        src = os.path.join(b.CSRC, "linear_mma_w%d.cu" % w)
        cmd = [nvcc] + b.ARCH + b.NVCC_FLAGS + ["-Xptxas", "-v", "-c", src, "-o", str(out / ("w%d.o" % w))]
        procs[w] = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    text = {}
    for w, p in procs.items():
        text[w] = p.communicate()[0]
        assert p.returncode == 0, text[w][-2000:]
    return text


def spills(report):
    """(kernel, spill store bytes, spill load bytes) for every linear kernel entry."""
    out, cur = [], None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur and "trellis_linear_" in cur:
            out.append((cur, int(m.group(1)), int(m.group(2))))
            cur = None
    return out


@pytest.mark.parametrize("w", WIDTHS)
def test_linear_kernels_do_not_spill(reports, w):
    entries = spills(reports[w])
    assert any("tc_kernel" in k for k, _, _ in entries), "no tcgen05 kernel in the %d-bit report" % w
    bad = [(k, st, ld) for k, st, ld in entries if st or ld]
    assert not bad, "spills at %d bits: %s" % (w, bad)


def test_the_spill_reader_sees_a_spill():
    """Control: the reader finds a spill in a report that has one."""
    report = ("ptxas info    : Compiling entry function '_ZN3tfx24trellis_linear_tc_kernelILi4EEEvv' for 'sm_103a'\n"
              "ptxas info    : Used 64 registers, 72 bytes spill stores, 72 bytes spill loads\n")
    assert spills(report) == [("_ZN3tfx24trellis_linear_tc_kernelILi4EEEvv", 72, 72)]
