"""Runs one workload through the library a few times, for profiler captures.

    python -m scaled_dot_product_gb300.profile_case --workload 2 [--batch B] [--rope]
        [--qk-mode M] [--iters K]
    python -m scaled_dot_product_gb300.profile_case --rotary [--iters K]
    python -m scaled_dot_product_gb300.profile_case --workload 3 --backward [--iters K]

Inputs are the seeded synthetic workloads of scaled_dot_product_gb300.workloads; every
launch goes through the C ABI (libsdpa.so).  Prints the kernel names and the status word.
"""
from __future__ import annotations

import argparse

import torch

from . import sdpa
from .workloads import WORKLOADS, as4d, draw_dy, make_rotary_inputs, rope_caches, workload


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--rope", action="store_true", help="rotate Q and the new K rows first")
    ap.add_argument("--qk-mode", type=int, default=None, help="also write the qk output at this stage")
    ap.add_argument("--rotary", action="store_true", help="standalone rotary (bf16, B=4, S=4096, 32 x 128)")
    ap.add_argument("--backward", action="store_true", help="the backward (sdpa_attn_bwd) of the workload")
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()
    torch.cuda.set_device(0)
    if a.rotary:
        ri = make_rotary_inputs(B=4, N=32, S=4096, D=128, dtype=torch.bfloat16, layout="bsnh", cache="ids",
                                max_pos=8192, seed=7).to("cuda")
        y = torch.empty_like(ri.x)
        for _ in range(a.iters):
            sdpa.sdpa_rotary(ri.x, ri.cos, ri.sin, ri.position_ids, num_heads=32, y=y)
    elif a.backward:
        case_cpu = workload(a.workload, batch=a.batch)
        case = case_cpu.to("cuda")
        q, k, v = case.views()
        dy = as4d(draw_dy(case_cpu, seed=3000 + a.workload).to("cuda"), case.q_layout, case.Nq)
        for _ in range(a.iters):
            sdpa.sdpa_attn_bwd(q, k, v, dy, **sdpa.case_kwargs(case))
    else:
        case = workload(a.workload, batch=a.batch)
        if a.rope:
            case.rotary_cos, case.rotary_sin = rope_caches(case.T, case.H // 2, case.dtype)
        case = case.to("cuda")
        op = "decode" if a.workload == 4 else "fwd"
        ws = sdpa.case_workspace(case, op)
        outs = sdpa.case_outputs(case)
        extra = {}
        if a.qk_mode is not None:
            extra = dict(qk_out=torch.empty(case.B, case.Nq, case.S, case.T, dtype=torch.float32, device="cuda"),
                         qk_mode=a.qk_mode)
        for _ in range(a.iters):
            sdpa.run_case(case, op, outputs=outs, workspace=ws, **extra)
    torch.cuda.synchronize()
    print("kernel", sdpa.sdpa_last_kernel_name(), "status", sdpa.sdpa_query_status())


if __name__ == "__main__":
    main()
