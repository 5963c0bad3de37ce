"""Register and stack use of every kernel, from ptxas's resource report
(-Xptxas -v) of a build for sm_103a: no kernel spills registers, except the
decode kernel's H = 4096 instance, whose 512-thread blocks cap it at 128
registers (it keeps a few words of its wider input rows on the stack; the
H = 2048 instance the benchmark runs does not).  A regression here costs
memory traffic inside the hot loops, so it fails the build check rather than
showing up later as a slower kernel."""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int4_grouped_gemm_gb300", "csrc")
ALLOWED_SPILL = {"decode_stack_kernelILi4096E": 160}  # bytes of spill stores


def _report(src):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I" + os.path.join(ROOT, "include"), "-Xptxas", "-v", "-c", os.path.join(CSRC, src),
                        "-o", os.devnull], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stderr


def test_no_register_spills():
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("no nvcc")
    sources = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    with ThreadPoolExecutor(max_workers=len(sources)) as ex:
        reports = dict(zip(sources, ex.map(_report, sources)))
    seen = 0
    for src, text in reports.items():
        fn = None
        for line in text.splitlines():
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                fn = m.group(1)
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and fn:
                seen += 1
                stores = int(m.group(1))
                limit = next((v for k, v in ALLOWED_SPILL.items() if k in fn), 0)
                assert stores <= limit, f"{src}: {fn} spills {stores} bytes (allowed {limit})"
    assert seen >= 15  # every kernel of the library was reported


def test_attention_kernel_leaves_room_for_the_merge_block():
    """The GQA attention kernel (one 256-thread block per SM) uses few
    enough registers that a block of the merge kernel (a programmatic
    dependent, 256 threads) fits beside it in the SM's 65,536 registers and
    is resident before the attention blocks finish (at 209 registers it was
    not, and the 32K call took 3 us longer)."""
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("no nvcc")
    text = _report("attention.cu")
    regs, fn = {}, None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            fn = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and fn:
            regs[fn] = int(m.group(1))
    attn = {f: r for f, r in regs.items() if "gqa_attention_kernel" in f}
    merge = [r for f, r in regs.items() if "gqa_combine_kernel" in f]
    assert len(attn) == 2 and len(merge) == 1, regs
    for f, r in attn.items():
        # registers are allocated per warp in units of 256 (8 per thread)
        per_block = lambda n: 256 * ((n + 7) // 8 * 8)  # noqa: E731
        assert per_block(r) + per_block(merge[0]) <= 65536, (f, r, merge[0])
