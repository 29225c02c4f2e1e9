"""The bounds-checking debug build (libsdpa_bounds.so, compiled with -DSDPA_BOUNDS_CHECK).

In that build the kernels range-check the indices of their global loads and stores, TMA
coordinates and staging offsets; a failed check records its site and skips the access, and
sdpa_query_status reports SDPA_ERR_BOUNDS (no trap, no fault).  On valid problems no check
may fire and the results must equal the oracle's, exactly as with the normal build.  The
library runs in a fresh process, so that it never shares one with libsdpa.so.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
from scaled_dot_product_gb300 import build, sdpa
sdpa.LIB_PATH = build.build(bounds_check=True)
import oracle
from oracle_adapter import expected_present, problem
from scaled_dot_product_gb300.workloads import as4d, make_case, workload
TOL = {{torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}}
cases = [
    (workload(2, small=True), "fwd"),    # softcap, fixed maximum, nonpad
    (workload(3, small=True), "fwd"),    # window, sink, seqlens_k
    (workload(5, small=True), "fwd"),    # additive mask, rank-4 K/V, q bias
    (workload(6, small=True), "fwd"),    # binary keep mask
    (workload(1), "fwd"),                # fp32: the general kernel
    (workload(4, small=True), "decode"), # split-KV decode with present
    (make_case("past_present", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=40, L=40, P=70, H=64, seed=5,
               causal="lower_right", want_present=True), "fwd"),   # kv_concat + tensor cores
]
names = set()
for c, op in cases:
    d = c.to("cuda")
    y, pk, pv = sdpa.run_case(d, op, workspace=sdpa.case_workspace(d, op))
    torch.cuda.synchronize()
    names.add(sdpa.sdpa_last_kernel_name())
    rc = sdpa.sdpa_query_status()
    assert rc == sdpa.SDPA_OK, (c.name, rc, sdpa.sdpa_last_error())
    got = as4d(y.float().cpu(), c.q_layout, c.Nq).double().numpy()
    err = np.abs(got - oracle.attention(problem(c))).max()
    assert err <= TOL[c.dtype], (c.name, err)
    if c.want_present:
        ek, ev = expected_present(c)
        bits = torch.int16 if c.dtype != torch.float32 else torch.int32
        assert torch.equal(pk.cpu().view(bits), ek.view(bits)) and torch.equal(pv.cpu().view(bits), ev.view(bits))
print("kernels", sorted(names))
"""


def test_bounds_checking_build_runs_clean_on_valid_problems():
    script = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "prefill_tc" in r.stdout and "decode_splitkv" in r.stdout and "simt_fwd" in r.stdout, r.stdout
