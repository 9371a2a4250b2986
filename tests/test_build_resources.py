"""Build-time resource checks from ptxas's report (no GPU).

"Tiled matrix multiplication" ("Pitfalls"): register spills from oversized
thread tiles turn into local-memory traffic.  Every kernel of the library
must compile without spills, within the register count its launch allows.
"""
import os
import re

from dense_gemm_12_gb300 import _build


def _report(gemm_lib):
    path = os.path.join(_build.BUILD_DIR, "ptxas.log")
    if not os.path.exists(path):
        _build.build(force=True)
    return open(path).read()


def _functions(text):
    """(mangled name, properties text) per compiled entry function."""
    out = []
    for m in re.finditer(r"Function properties for (\S+)\n(.*?)(?=\nptxas info\s+: Used)", text,
                         flags=re.S):
        out.append((m.group(1), m.group(2)))
    return out


def test_no_kernel_spills(gemm_lib):
    text = _report(gemm_lib)
    funcs = _functions(text)
    assert len(funcs) >= 10, "expected every kernel in the report"
    spilling = []
    for name, props in funcs:
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", props)
        assert m, name
        if int(m.group(1)) or int(m.group(2)):
            spilling.append((name, m.group(0)))
    assert not spilling, spilling


def test_register_counts_fit_the_launches(gemm_lib):
    # 192-thread tcgen05 kernels and 224-thread decode kernel: at most 255
    # registers; the 384-thread CUDA-core kernel launches at 168 (setmaxnreg
    # moves registers between its warpgroups at run time)
    text = _report(gemm_lib)
    for m in re.finditer(r"Compiling entry function '(\S+)'.*?Used (\d+) registers", text,
                         flags=re.S):
        name, regs = m.group(1), int(m.group(2))
        assert regs <= 255, (name, regs)
        if "simt_gemm_kernel" in name:
            assert regs <= 168, (name, regs)
