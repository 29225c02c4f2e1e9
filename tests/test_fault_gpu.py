"""Failure detection without faulting the GPU: every barrier wait of the tensor-core
kernel is time-bounded.  With the limit forced to 1 ns (SDPA_WAIT_LIMIT_NS, read once per
process), the first wait that is not already satisfied expires: the kernel raises its
abort flag, lets its own copies and MMAs finish, frees its tensor memory and records
SDPA_ERR_TIMEOUT, which sdpa_query_status reports.  The context must stay usable."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, torch
    sys.path.insert(0, {root!r})
    from scaled_dot_product_gb300 import sdpa
    from scaled_dot_product_gb300.workloads import workload
    case = workload(2, small=True).to("cuda")
    y, _, _ = sdpa.run_case(case, "fwd")
    rc = sdpa.sdpa_query_status()
    print("KERNEL", sdpa.sdpa_last_kernel_name())
    print("STATUS", rc)
    # the context is still usable: a plain copy and a second status read succeed
    z = torch.arange(1024, device="cuda").sum().item()
    print("AFTER", z, sdpa.sdpa_query_status())
""")


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())


def test_expired_waits_report_timeout_and_leave_the_context_usable():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from scaled_dot_product_gb300 import build
    build.build()
    out = _run({"SDPA_WAIT_LIMIT_NS": "1"})
    assert out["KERNEL"].startswith("prefill_tc")
    assert int(out["STATUS"]) == 9                     # SDPA_ERR_TIMEOUT
    assert out["AFTER"].split() == [str(sum(range(1024))), "0"]


def test_default_limit_runs_clean():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    out = _run({})
    assert int(out["STATUS"]) == 0
