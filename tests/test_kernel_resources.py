"""Register and spill budgets of the hot-path kernels, checked at compile time on
the CPU (ptxas -v for sm_103a; no GPU needed).

These are the figures the kernels were measured with: the projection's
across-heads instantiation fits its 10-warp block in 168 registers with no
spills, and the pipelined norm/RoPE and KV-cache kernels and the row
quantiser spill nothing.  A change that pushes a kernel past its budget fails
here, before any GPU time is spent on it.
"""
import concurrent.futures as cf
import os
import re
import subprocess

import pytest

from rope_attention_gb300 import build

CSRC = build.CSRC

# kernel name -> (max registers, max spill-store bytes), for every instantiation
BUDGETS = {
    "qkv_project.cu": {
        "qkv_project_kernelILi0E": (168, 0),      # across heads: the 720p step's kernel
        "qkv_project_kernelILi128E": (168, 16),   # per-head norm, head_dim 128 (8 bytes today)
        "qkv_project_kernelILi64E": (168, 64),    # per-head norm, head_dim 64 (32 bytes today)
    },
    "qk_norm_rope.cu": {
        "qk_norm_rope_staged_kernel": (128, 0),
        "qk_norm_rope_nbsd_kernel": (75, 0),      # 288 threads, 3 blocks per SM: at most 75 registers
        "qk_norm_rope_kernel": (128, 0),
    },
    "kv_cache.cu": {
        "kv_staged_kernel": (128, 0),
    },
    "row_quant.cu": {
        "row_quant": (255, 0),
    },
}

ENTRY = re.compile(r"Compiling entry function '([^']+)'")
SPILL = re.compile(r"(\d+) bytes spill stores")
REGS = re.compile(r"Used (\d+) registers")


def ptxas_report(src: str, tmpdir: str) -> dict[str, tuple[int, int]]:
    obj = os.path.join(tmpdir, src + ".o")
    cmd = [build.nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", *build.ARCH,
           "-I", build.INCLUDE, "-I", CSRC, "-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out, name, spill = {}, None, 0
    for ln in r.stderr.splitlines():
        m = ENTRY.search(ln)
        if m:
            name, spill = m.group(1), 0
            continue
        m = SPILL.search(ln)
        if m and name:
            spill = int(m.group(1))
        m = REGS.search(ln)
        if m and name:
            out[name] = (int(m.group(1)), spill)
            name = None
    return out


@pytest.fixture(scope="module")
def reports(tmp_path_factory):
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    tmp = str(tmp_path_factory.mktemp("ptxas"))
    with cf.ThreadPoolExecutor(max_workers=len(BUDGETS)) as ex:
        futs = {src: ex.submit(ptxas_report, src, tmp) for src in BUDGETS}
        return {src: f.result() for src, f in futs.items()}


@pytest.mark.parametrize("src", sorted(BUDGETS))
def test_kernels_within_register_and_spill_budget(reports, src):
    rep = reports[src]
    for kernel, (max_regs, max_spill) in BUDGETS[src].items():
        hits = {name: v for name, v in rep.items() if kernel in name}
        assert hits, f"{kernel}: no such entry in {src} (ptxas saw {sorted(rep)})"
        for name, (regs, spill) in hits.items():
            assert regs <= max_regs, f"{name}: {regs} registers > {max_regs}"
            assert spill <= max_spill, f"{name}: {spill} bytes of spill stores > {max_spill}"
