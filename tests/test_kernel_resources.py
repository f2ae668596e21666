"""Register budgets of the hot kernels, checked at compile time on the CPU.

The design fixes how many CTAs share an SM, and so how many registers a
thread may use: the small-M kernels with one or two rows per pass run two
256-thread CTAs per SM (at most 128 registers), the eight-row form one CTA;
the tensor-core MoE kernel runs one 544-thread CTA (at most 96: five of its
17 warps share one of the SM's four sub-partitions, whose register files hold
16,384 registers each); the tiled router
runs two 256-thread blocks (at most 128).  The launch bounds make the compiler
keep those limits, but it does so by spilling to local memory, which nothing
else would notice: this test compiles the translation units with ptxas'
resource report and fails on any spill or any kernel over its budget.
"""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from group_quantized_moe_gb300 import build_lib

UNITS = ["smallm_one.cu", "smallm_lo.cu", "smallm_hi.cu", "moe_tc.cu", "router.cu"]
ENTRY = re.compile(r"Compiling entry function '(\w+)'")
SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
REGS = re.compile(r"Used (\d+) registers")
# Off the measured path, and known to spill a word: the top-k variants for
# more than 256 experts (their per-lane logit array is indexed at run time)
# and the one-block dispatch (prefill only, latency-bound).
SPILL_EXEMPT = ("router_topk_kernelILi16EE", "router_topk_kernelILi32EE", "moe_dispatch_kernel")


def _budget(name: str):
    m = re.search(r"smallm_kernelILi\d+ELi\d+ELi\d+ELi\d+ELb[01]ELi(\d+)E", name)
    if m:
        return ("small-M, %s row(s) per pass" % m.group(1), 128 if int(m.group(1)) <= 2 else 255)
    if "moe_tc_kernel" in name:
        return ("tensor-core MoE", 96)
    m = re.search(r"router_logits_tiled_kernelILb[01]ELi(\d+)EE", name)
    if m:
        return ("tiled router", 128 if int(m.group(1)) <= 8 else 255)
    return (None, 255)


def _report(unit: str, out_dir: str) -> str:
    cmd = [build_lib._nvcc(), *build_lib.ARCH, *build_lib.FLAGS, "-Xptxas", "-v", "-c",
           os.path.join(build_lib.CSRC, unit), "-o", os.path.join(out_dir, unit + ".o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return r.stdout + r.stderr


def test_hot_kernels_fit_their_register_budget_without_spills(tmp_path):
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not found")
    with ThreadPoolExecutor(len(UNITS)) as ex:
        reports = list(ex.map(lambda u: _report(u, str(tmp_path)), UNITS))
    seen, problems = 0, []
    for unit, text in zip(UNITS, reports):
        name = None
        for line in text.splitlines():
            m = ENTRY.search(line)
            if m:
                name = m.group(1)
                continue
            if name is None:
                continue
            m = SPILL.search(line)
            if m and (int(m.group(1)) or int(m.group(2))) and not any(x in name for x in SPILL_EXEMPT):
                problems.append(f"{unit}: {name} spills ({line.strip()})")
            m = REGS.search(line)
            if m:
                what, limit = _budget(name)
                if what:
                    seen += 1
                    if int(m.group(1)) > limit:
                        problems.append(f"{unit}: {what} kernel {name} uses {m.group(1)} "
                                        f"registers, budget {limit}")
                name = None
    assert seen >= 30, f"only {seen} budgeted kernels found in the reports"
    assert not problems, "\n".join(problems)
