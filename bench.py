"""Benchmark of the attention forward path on GB300.

Default: the GQA prefill workload (bf16, B=2, S=T=2048, 32 query / 8 kv heads, H=128,
upper-left causal, softcap 30, nonpad lengths in [1024, 2048]) at N=1, printed as ONE
JSON line on rank 0.  The other workloads are measured in the same run and reported under
"secondary" (decode in KV GB/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
  python bench.py --profile-run --workload W [--batch B] [--rope] [--qk-mode M] [--iters K]
  python bench.py --profile-run --rotary | --backward --workload 3 [--iters K]

--impl reference times the double-precision CPU oracle (the only other program this
repository has for the same computation) on bounded samples of the same workload.
Under torchrun (N > 1) every rank runs an independent replica of the workload on its
own GPU (the path needs no exchange between GPUs; scaling is weak).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from scaled_dot_product_gb300.workloads import WORKLOADS, Case, workload  # noqa: E402

L2_FLUSH_BYTES = 256 << 20          # larger than the 129 MB L2


# ------------------------------------------------------------------------------ work model

def admitted_pairs_per_row(case: Case) -> np.ndarray:
    """(B, S) count of keys each query row must attend under the structural rules
    (causal, window, nonpad / seqlens_k exclusion).  Float masks and filter values exclude
    nothing, so every such key counts as work."""
    T = case.T
    out = np.zeros((case.B, case.S), dtype=np.int64)
    lens = case.lens.cpu().numpy().astype(np.int64) if case.lens is not None else None
    i = np.arange(case.S, dtype=np.int64)
    for b in range(case.B):
        hi = np.full(case.S, T - 1, dtype=np.int64)
        lo = np.zeros(case.S, dtype=np.int64)
        if case.causal != "none":
            if case.causal == "upper_left":
                pos = i
            else:
                tv = lens[b] + 1 if case.len_kind == "seqlens_k" else T
                pos = tv - case.S + i
            hi = np.minimum(hi, pos)
            if case.window > 0:
                lo = np.maximum(lo, pos - case.window + 1)
        if case.len_kind == "nonpad":
            hi = np.minimum(hi, lens[b] - 1)
        elif case.len_kind == "seqlens_k":
            hi = np.minimum(hi, lens[b])
        out[b] = np.maximum(0, hi - lo + 1)
    return out


def prefill_flops(case: Case) -> float:
    return float(admitted_pairs_per_row(case).sum()) * case.Nq * 2.0 * (case.H + case.Hv)


def decode_bytes(case: Case) -> float:
    es = torch.tensor([], dtype=case.dtype).element_size()
    past = case.B * case.Nkv * case.P * (case.H + case.Hv) * es
    new = case.B * case.Nkv * case.L * (case.H + case.Hv) * es
    present = case.B * case.Nkv * case.T * (case.H + case.Hv) * es if case.want_present else 0
    qy = case.B * case.Nq * case.S * (case.H + case.Hv) * es
    return float(past + new + present + qy)


def decode_attended_bytes(case: Case) -> float:
    """The secondary decode figure: bytes of the K/V-cache rows the step actually attends
    (positions j < keylen[b] of every kv head), without the present copy."""
    es = torch.tensor([], dtype=case.dtype).element_size()
    T = case.T
    if case.lens is not None and case.len_kind in ("keylen", "nonpad"):
        keys = sum(min(int(n), T) for n in case.lens.tolist())
    elif case.lens is not None and case.len_kind == "seqlens_k":
        keys = sum(min(int(n) + 1, T) for n in case.lens.tolist())
    else:
        keys = case.B * T
    return float(keys * case.Nkv * (case.H + case.Hv) * es)


def is_decode(idx: int) -> bool:
    return idx == 4


# NVIDIA's GB300 dense BF16/FP16 tensor rate (per GPU, without 2:4 sparsity), the nominal
# figure the measured cuBLAS peak is compared with
NOMINAL_BF16_TFLOPS = 2250.0


def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the machine type)."""
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


# ------------------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# Sources each kernel family is built from: a traffic figure stays valid while they hash
# to the digest recorded with it.
KERNEL_SOURCES = {
    "prefill_tc": ("prefill_tc.cu", "prefill_tc.h", "tc_ptx.cuh", "common.cuh"),
    "decode_splitkv": ("decode.cu", "internal.h", "common.cuh"),
    "rotary": ("rotary.cu", "internal.h", "common.cuh"),
    "qk_tc": ("qk.cu", "prefill_tc.h", "tc_ptx.cuh", "common.cuh"),
    "bwd_tc": ("bwd_tc.cu", "prefill_tc.cu", "prefill_tc.h", "tc_ptx.cuh", "common.cuh", "internal.h"),
}


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/', re.S)


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments (string and character literals kept), with
    trailing blanks and blank lines dropped: what the compiler sees, for the digest."""
    code = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    lines = (ln.rstrip() for ln in code.splitlines())
    return "\n".join(ln for ln in lines if ln)


def source_digest(kernel: str, read=None) -> str:
    """Digest of the kernel family's sources without comments: counters taken on the sources
    stay valid through comment edits and are dropped on any code change.  `read(name)` returns
    a source's text (default: the working tree)."""
    fam = next((f for f in KERNEL_SOURCES if kernel.startswith(f)), None)
    csrc = os.path.join(ROOT, "scaled_dot_product_gb300", "csrc")
    names = KERNEL_SOURCES[fam] if fam else tuple(sorted(os.listdir(csrc)))
    if read is None:
        read = lambda n: open(os.path.join(csrc, n), encoding="utf-8").read()
    h = hashlib.sha256()
    for n in names:
        h.update(n.encode())
        h.update(strip_comments(read(n)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("source_digest") != source_digest(kernel):
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------ native arm

HOST_LEAD_CYCLES = 4_000_000       # ~2 ms of GPU sleep ahead of the timed steps


def time_device(fn, steps, warmup, flush_buf, barrier):
    """CUDA-event times of `steps` calls of fn on the current stream (L2 flushed before each
    when flush_buf is given, outside the events).  The flush buffer is written once before the
    warm-ups (its first write maps fresh pages and slows the kernel that follows it), and a
    short device-side sleep is queued ahead of the first timed step, so that the host has
    enqueued the first steps before the GPU reaches them: an event pair then brackets device
    work only, never the GPU idling while the host prepares a call."""
    if flush_buf is not None:
        flush_buf.fill_(0)              # first touch of the flush buffer outside the timed region
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    torch.cuda._sleep(HOST_LEAD_CYCLES)
    for s in range(steps):
        if flush_buf is not None:
            flush_buf.fill_(s & 0xff)       # evict the inputs from L2 between timed steps
        starts[s].record()
        fn()
        ends[s].record()
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return ms, wall


def with_rope(case: Case) -> Case:
    """The same case with GroupQueryAttention's rotary step on Q and the new K rows
    (rank-2 cos/sin tables of T rows over all H channels)."""
    from scaled_dot_product_gb300.workloads import rope_caches
    case.rotary_cos, case.rotary_sin = rope_caches(case.T, case.H // 2, case.dtype)
    case.name += "_rope"
    return case


def measure_native(idx: int, steps: int, warmup: int, barrier, with_e2e: bool = True, batch=None,
                   rope: bool = False, qk_mode=None):
    from scaled_dot_product_gb300 import sdpa
    case_cpu = workload(idx, batch=batch)
    if rope:
        case_cpu = with_rope(case_cpu)
    case = case_cpu.to("cuda")
    op = "decode" if is_decode(idx) else "fwd"
    ws = sdpa.case_workspace(case, op)
    outs = sdpa.case_outputs(case)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    extra = {}
    if qk_mode is not None:
        extra = dict(qk_out=torch.empty(case.B, case.Nq, case.S, case.T, dtype=torch.float32, device="cuda"),
                     qk_mode=qk_mode)
    run = lambda: sdpa.run_case(case, op, outputs=outs, workspace=ws, **extra)
    run()
    torch.cuda.synchronize()
    kernel = sdpa.sdpa_last_kernel_name()
    n0 = sdpa.sdpa_launch_count()
    run()
    torch.cuda.synchronize()
    per_step_launches = sdpa.sdpa_launch_count() - n0
    input_bytes = case.input_bytes()
    use_flush = input_bytes < (129 << 20)
    with ClockSampler(torch.cuda.current_device()) as clk:
        ms, wall = time_device(run, steps, warmup, flush if use_flush else None, barrier)
    res = {"idx": idx, "case": case_cpu, "op": op, "kernel": kernel, "ms": ms, "wall": wall,
           "launches": per_step_launches * steps, "clocks": clk.summary(), "l2_flush": use_flush}

    if with_e2e:
        res.update(measure_e2e(case_cpu, case, outs, ws, op, steps, barrier, extra))
    return res


E2E_INPUTS = ("q", "k", "v", "past_k", "past_v", "q_bias", "k_bias", "v_bias", "head_sink", "add_mask",
              "keep_mask", "lens")


def measure_e2e(case_cpu, case, outs, ws, op, steps, barrier, extra):
    """End to end through the C ABI with host buffers.  Every step uploads all of its inputs
    from pinned host memory, runs the kernels and reads every output back to pinned host
    memory, all inside the timed region.  Steps are pipelined as a serving loop runs them:
    two device buffer sets, the upload of step k+1 (copy stream) and the read-back of step
    k-1 (another copy stream) overlap the kernels of step k; events keep a set's inputs until
    its kernels have read them and its outputs until they are read back.  The value is K
    steps over one timed region, from the first upload to the last read-back."""
    from scaled_dot_product_gb300 import sdpa
    case2 = case_cpu.to("cuda")
    sets = [(case, outs, ws), (case2, sdpa.case_outputs(case2), sdpa.case_workspace(case2, op))]
    host_in = {n: getattr(case_cpu, n).contiguous().pin_memory() for n in E2E_INPUTS
               if getattr(case_cpu, n) is not None}
    dev_out = [[o[0]] + [t for t in o[2:] if t is not None] for _, o, _ in sets]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d] for d in dev_out]
    h2d = sum(h.numel() * h.element_size() for h in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    run_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def pipeline(n):
        for k in range(n):
            i = k & 1
            c, o, w = sets[i]
            if k >= 2:
                s_in.wait_event(run_done[i])          # step k-2's kernels have read set i
            with torch.cuda.stream(s_in):
                for name, h in host_in.items():
                    getattr(c, name).copy_(h, non_blocking=True)
                in_done[i].record(s_in)
            s_run.wait_event(in_done[i])
            if k >= 2:
                s_run.wait_event(out_done[i])         # step k-2's outputs have been read back
            with torch.cuda.stream(s_run):
                sdpa.run_case(c, op, outputs=o, workspace=w, **extra)
                run_done[i].record(s_run)
            s_out.wait_event(run_done[i])
            with torch.cuda.stream(s_out):
                for hd, dd in zip(host_out[i], dev_out[i]):
                    hd.copy_(dd, non_blocking=True)
                out_done[i].record(s_out)

    n = max(6, min(steps, 50))
    pipeline(4)                                       # warm-up
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_run.wait_event(t0)
    s_out.wait_event(t0)
    pipeline(n)
    t1.record(s_out)                                  # the last read-back ends after everything
    torch.cuda.synchronize()
    barrier()
    return dict(e2e_ms=[t0.elapsed_time(t1) / n], h2d=h2d, d2h=d2h, e2e_steps=n)


ROTARY_SHAPE = dict(B=4, N=32, S=4096, D=128)     # packed (B, S, N*D) bf16, 128 MiB in and out


def rotary_bytes(B, N, S, D, esize, R=None):
    """Algorithmic bytes of one standalone rotary call: x read, y written, one int64
    position id and one cos and one sin row (R/2 entries) per (b, s)."""
    R = D if R is None else R
    return 2 * B * N * S * D * esize + B * S * 8 + 2 * B * S * (R // 2) * esize


def measure_rotary(steps: int, warmup: int, barrier, hbm: float):
    from scaled_dot_product_gb300 import sdpa
    from scaled_dot_product_gb300.workloads import make_rotary_inputs
    sh = ROTARY_SHAPE
    ri = make_rotary_inputs(dtype=torch.bfloat16, layout="bsnh", cache="ids", max_pos=2 * sh["S"],
                            seed=7, **sh).to("cuda")
    y = torch.empty_like(ri.x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    run = lambda: sdpa.sdpa_rotary(ri.x, ri.cos, ri.sin, ri.position_ids, num_heads=sh["N"], y=y)
    run()
    torch.cuda.synchronize()
    n0 = sdpa.sdpa_launch_count()
    ms, _ = time_device(run, steps, warmup, flush, barrier)
    launches = sdpa.sdpa_launch_count() - n0
    m = statistics.mean(ms)
    gbs = rotary_bytes(sh["B"], sh["N"], sh["S"], sh["D"], 2) / (m * 1e-3) / 1e9
    return {"workload": "rotary_bf16_b4_s4096_n32_d128_position_ids", "value": gbs, "unit": "GB/s",
            "ms_per_step": m, "kernel": "rotary", "gpu_launches": launches,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "traffic": ncu_traffic("rotary")}, "l2_flush": True}


def backward_flops(case: Case) -> float:
    """Algorithmic work of the backward (the GroupQueryAttention gradient graph): per admitted
    (query, key) pair the score recompute Q K^T (2H), dP = dY V^T (2Hv), dQ = dS K (2H),
    dK = dS^T Q (2H) and dV = P^T dY (2Hv), i.e. 2.5 times the forward's 2(H + Hv)."""
    return float(admitted_pairs_per_row(case).sum()) * case.Nq * 2.0 * (3 * case.H + 2 * case.Hv)


def measure_backward(idx: int, steps: int, warmup: int, barrier, tfl, tfl_src):
    """Backward (sdpa_attn_bwd) on a workload: inputs and dY resident, dQ / dK / dV written
    every step; L2 flushed between timed steps."""
    from scaled_dot_product_gb300 import sdpa
    from scaled_dot_product_gb300.workloads import as4d, draw_dy
    case_cpu = workload(idx)
    case = case_cpu.to("cuda")
    q, k, v = case.views()
    dy = as4d(draw_dy(case_cpu, seed=3000 + idx).to("cuda"), case.q_layout, case.Nq)
    kw = sdpa.case_kwargs(case)
    dq = torch.empty(case.B, case.Nq, case.S, case.H, dtype=case.dtype, device="cuda")
    dk = torch.empty(case.B, case.Nkv, case.T, case.H, dtype=case.dtype, device="cuda")
    dv = torch.empty(case.B, case.Nkv, case.T, case.Hv, dtype=case.dtype, device="cuda")
    params, keep = sdpa.make_params(q, k, v, **kw)
    ws = torch.empty(sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_BWD), dtype=torch.uint8, device="cuda")
    run = lambda: sdpa.sdpa_attn_bwd(q, k, v, dy, dq=dq, dk=dk, dv=dv, workspace=ws, **kw)
    run()
    torch.cuda.synchronize()
    kernel = sdpa.sdpa_last_kernel_name()
    n0 = sdpa.sdpa_launch_count()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    with ClockSampler(torch.cuda.current_device()) as clk:
        ms, _ = time_device(run, steps, warmup, flush, barrier)
    launches = sdpa.sdpa_launch_count() - n0
    m = statistics.mean(ms)
    tf = backward_flops(case_cpu) / (m * 1e-3) / 1e12
    return {"workload": case_cpu.name + "_backward", "value": tf, "unit": "TFLOP/s", "ms_per_step": m,
            "work_per_step": f"{backward_flops(case_cpu):.4g} flop (2.5x the forward's)",
            "kernel": kernel, "gpu_launches": launches, "launches_per_step": launches // max(1, steps + warmup),
            "roofline": {"bound": "tensor", "achieved": tf, "peak": tfl, "unit": "TFLOP/s", "frac": tf / tfl,
                         "peak_source": f"{tfl_src} bf16 dense burst", "traffic": ncu_traffic(kernel)},
            "l2_flush": True, "clocks": clk.summary()}


def metric_of(idx: int, case: Case, ms: float):
    if is_decode(idx):
        return decode_bytes(case) / (ms * 1e-3) / 1e9, "GB/s"
    return prefill_flops(case) / (ms * 1e-3) / 1e12, "TFLOP/s"


def roofline(idx: int, case: Case, res: dict, hbm, tfl, tfl_src):
    ms = statistics.mean(res["ms"])
    if is_decode(idx):
        achieved = decode_bytes(case) / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": f"{tfl_src} copy bandwidth",
                "traffic": ncu_traffic(res["kernel"]),
                "attended_kv_GBps": decode_attended_bytes(case) / (ms * 1e-3) / 1e9}
    achieved = prefill_flops(case) / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": tfl, "unit": "TFLOP/s",
            "frac": achieved / tfl, "peak_source": f"{tfl_src} bf16 dense burst",
            "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
            "nominal_peak": f"{NOMINAL_BF16_TFLOPS:.0f} TFLOP/s dense bf16 (NVIDIA GB300 figure)",
            "traffic": ncu_traffic(res["kernel"])}


# ------------------------------------------------------------------------------ oracle arm

class OracleSampler:
    """Times the oracle on samples of query rows of one workload (CPU baseline / reference
    arm).  The per-row cost is calibrated once, so every step can be sized from a budget."""

    def __init__(self, idx: int, case: Case = None):
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from oracle_adapter import problem
        self.oracle = oracle
        self.idx = idx
        self.case = case if case is not None else workload(idx)
        self.pr = problem(self.case)
        self.rng = np.random.default_rng(7)
        self.counts = admitted_pairs_per_row(self.case)
        t0 = time.perf_counter()
        _, self.threads = oracle.attention_rows(self.pr, self._rows(64))
        self.sec_per_row = max((time.perf_counter() - t0) / 64, 1e-7)

    def _rows(self, n):
        c = self.case
        return np.stack([self.rng.integers(0, c.B, n), self.rng.integers(0, c.Nq, n),
                         self.rng.integers(0, c.S, n)], -1).astype(np.int64)

    def step(self, target_s: float):
        c = self.case
        n = int(max(1, min(c.B * c.Nq * c.S, target_s / self.sec_per_row)))
        rows = self._rows(n)
        t0 = time.perf_counter()
        _, threads = self.oracle.attention_rows(self.pr, rows)
        secs = time.perf_counter() - t0
        if is_decode(self.idx):
            es = torch.tensor([], dtype=c.dtype).element_size()
            work = n * c.T * (c.H + c.Hv) * es        # KV-cache bytes the sampled rows read
            value, unit = work / secs / 1e9, "GB/s"
        else:
            work = float(self.counts[rows[:, 0], rows[:, 2]].sum()) * 2.0 * (c.H + c.Hv)
            value, unit = work / secs / 1e12, "TFLOP/s"
        return {"value": value, "unit": unit, "cores": threads, "cpu_model": cpu_model(), "kind": "oracle",
                "sample": f"{n} of {c.B * c.Nq * c.S} query rows of {c.name}, {secs:.2f} s on {threads} threads",
                "seconds": secs}


def oracle_sample(idx: int, target_s: float, case: Case = None):
    """One timed oracle sample of about target_s seconds (the CPU-baseline leg)."""
    return OracleSampler(idx, case).step(target_s)


# ------------------------------------------------------------------------------ main

def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (identity without a group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000,
                    help="timed steps (the default keeps nvidia-smi sampling inside the timed region)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work for the oracle baseline sample; 0 skips it")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size of the headline workload (profiling captures only)")
    ap.add_argument("--backward-only", action="store_true",
                    help="measure only the backward on the GQA workload (profiling captures)")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="total CPU time budget of the reference (oracle) arm")
    # profiler captures: run one case --iters times through the C ABI, untimed
    ap.add_argument("--profile-run", action="store_true",
                    help="run --workload (or --rotary / --backward) --iters times for a profiler capture, no timing")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--rope", action="store_true", help="--profile-run: rotate Q and the new K rows first")
    ap.add_argument("--qk-mode", type=int, default=None, help="--profile-run: also write the qk output at this stage")
    ap.add_argument("--rotary", action="store_true", help="--profile-run: the standalone rotary shape")
    ap.add_argument("--backward", action="store_true", help="--profile-run: the backward of --workload")
    a = ap.parse_args()
    if a.profile_run:
        profile_run(a)
        return
    warmup = max(3, a.warmup)
    idx = a.workload

    if a.impl == "reference":
        ws, rank, _ = dist_setup("gloo")
        if rank != 0:
            return
        sampler = OracleSampler(idx)
        case = sampler.case
        per_step = a.ref_seconds / (a.steps + warmup)
        for _ in range(warmup):
            sampler.step(per_step)
        vals, secs, last = [], [], None
        for _ in range(a.steps):
            last = sampler.step(per_step)
            vals.append(last["value"])
            secs.append(last["seconds"])
        value = statistics.mean(vals)
        line = {"impl": "reference", "metric": metric_name(idx), "value": value, "unit": last["unit"],
                "n_gpus": a.gpus, "steps": a.steps, "warmup": warmup,
                "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config_of(idx, case, None),
                "cpu_baseline": {"kind": "oracle", "cores": last["cores"], "sample": last["sample"],
                                 "value": value, "unit": last["unit"]},
                "e2e": {"value": value, "unit": last["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    ws, rank, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        barrier = lambda: dist.barrier()
    else:
        barrier = lambda: None
    from scaled_dot_product_gb300 import build as _b
    if rank == 0:
        _b.build()
    if ws > 1:
        barrier()
    hbm, tfl, tfl_sus, src = peaks()

    if a.backward_only:
        print(json.dumps(measure_backward(3, a.steps, warmup, barrier, tfl, src)))
        return
    res = measure_native(idx, a.steps, warmup, barrier, with_e2e=not a.no_e2e, batch=a.batch)
    case = res["case"]
    ms = statistics.mean(res["ms"])
    e2e_ms = statistics.mean(res["e2e_ms"]) if "e2e_ms" in res else float("nan")
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], device="cuda")
    value, unit = metric_of(idx, case, ms)
    e2e_value, _ = metric_of(idx, case, e2e_ms)
    if rank != 0:
        return
    line = {
        "metric": metric_name(idx), "value": value * ws, "unit": unit, "n_gpus": ws,
        "steps": a.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[case.dtype],
        "data": "synthetic (seeded, drawn in fp32 on the CPU, rounded once)",
        "config": config_of(idx, case, res),
        "kernel": res["kernel"],
        "ms_p10_p90": [float(np.percentile(res["ms"], 10)), float(np.percentile(res["ms"], 90))],
        "ms_median": float(np.median(res["ms"])),
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "e2e": ({"value": e2e_value * ws, "unit": unit, "h2d_bytes_per_step": res["h2d"],
                 "d2h_bytes_per_step": res["d2h"], "ms_per_step": e2e_ms, "steps": res["e2e_steps"],
                 "mode": "pipelined: the upload of step k+1 and the read-back of step k-1 overlap "
                         "step k (two device buffer sets, three streams); every step's copies are "
                         "inside the timed region"} if "e2e_ms" in res else None),
        "roofline": roofline(idx, case, res, hbm, tfl, src),
        "wall_s_timed_region": res["wall"],
    }
    if ws == 1 and a.cpu_seconds > 0:
        line["cpu_baseline"] = {k: v for k, v in oracle_sample(idx, a.cpu_seconds, case).items()
                                if k != "seconds"}
    if not a.no_secondary:
        # the other workloads and the NEXT rows, compact and last on the line, so that a
        # reader keeping only the line's tail still sees them:
        #   secondary [workload, value, unit, ms per step, roofline fraction, kernel]
        sec, sec_ms = [], {}
        for j in sorted(WORKLOADS):
            if j == idx:
                continue
            r = measure_native(j, max(5, min(a.steps // 2, 200)), warmup, barrier, with_e2e=False)
            m = statistics.mean(r["ms"])
            v, u = metric_of(j, r["case"], m)
            rf = roofline(j, r["case"], r, hbm, tfl, src) if j != 1 else None
            entry = [r["case"].name, round(v, 2), u, round(m, 5), None if rf is None else round(rf["frac"], 4), r["kernel"]]
            if rf is not None and "attended_kv_GBps" in rf:
                entry.append({"attended_kv_GBps": round(rf["attended_kv_GBps"], 1)})
            sec.append(entry)
            sec_ms[j] = m
            del r
            torch.cuda.empty_cache()
        # rotary [workload, value, unit, ms per step, overhead against the same workload
        # without the rotation (ms)]: standalone, and as the prologue of the GQA prefill and
        # of the decode step
        rot = measure_rotary(max(20, min(a.steps, 500)), warmup, barrier, hbm)
        nxt = [[rot["workload"], round(rot["value"], 1), rot["unit"], round(rot["ms_per_step"], 5), None]]
        for j in (2, 4):
            r = measure_native(j, max(5, min(a.steps // 2, 200)), warmup, barrier, with_e2e=False, rope=True)
            m = statistics.mean(r["ms"])
            v, u = metric_of(j, r["case"], m)
            base_ms = ms if j == idx else sec_ms.get(j)
            nxt.append([r["case"].name, round(v, 2), u, round(m, 5), None if base_ms is None else round(m - base_ms, 5)])
            del r
            torch.cuda.empty_cache()
        # backward [workload, value, unit, ms per step, roofline fraction, launches per step]
        bw = measure_backward(3, max(5, min(a.steps // 2, 100)), warmup, barrier, tfl, src)
        torch.cuda.empty_cache()
        # qk output [workload, ms per step, added ms, GB/s of qk output over the added time,
        # fraction of HBM]: qk_matmul_output_mode 0 and 3 on the GQA prefill
        qkl = []
        if idx == 2:
            for mode in (0, 3):
                r = measure_native(2, max(5, min(a.steps // 2, 200)), warmup, barrier, with_e2e=False, qk_mode=mode)
                m = statistics.mean(r["ms"])
                c = r["case"]
                out_bytes = c.B * c.Nq * c.S * c.T * 4
                extra_ms = m - ms
                gbs = out_bytes / (extra_ms * 1e-3) / 1e9 if extra_ms > 0 else None
                qkl.append([c.name + f"_qk_mode{mode}", round(m, 5), round(extra_ms, 5),
                            None if gbs is None else round(gbs, 1), None if gbs is None else round(gbs / hbm, 4)])
                del r
                torch.cuda.empty_cache()
        line["rotary"] = nxt
        line["backward"] = [[bw["workload"], round(bw["value"], 2), bw["unit"], round(bw["ms_per_step"], 5),
                             round(bw["roofline"]["frac"], 4), bw["launches_per_step"]]]
        if qkl:
            line["qk_output"] = qkl
        line["secondary"] = sec
    print(json.dumps(line))


def profile_run(a):
    """Runs one case a.iters times through the C ABI (for ncu captures; nothing is timed) and
    prints the kernel name and the device status word."""
    from scaled_dot_product_gb300 import build as _b, sdpa
    from scaled_dot_product_gb300.workloads import as4d, draw_dy, make_rotary_inputs, rope_caches
    _b.build()
    torch.cuda.set_device(0)
    if a.rotary:
        sh = ROTARY_SHAPE
        ri = make_rotary_inputs(dtype=torch.bfloat16, layout="bsnh", cache="ids", max_pos=2 * sh["S"], seed=7,
                                **sh).to("cuda")
        y = torch.empty_like(ri.x)
        for _ in range(a.iters):
            sdpa.sdpa_rotary(ri.x, ri.cos, ri.sin, ri.position_ids, num_heads=sh["N"], y=y)
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
        op = "decode" if is_decode(a.workload) else "fwd"
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


def metric_name(idx: int) -> str:
    if is_decode(idx):
        return "attention KV-cache GB/s (decode) vs GB300 HBM roofline"
    return "attention TFLOP/s (prefill) vs GB300 dense tensor-core roofline"


def config_of(idx: int, case: Case, res):
    c = {"workload": case.name, "B": case.B, "Nq": case.Nq, "Nkv": case.Nkv, "S": case.S,
         "T": case.T, "H": case.H, "causal": case.causal, "window": case.window,
         "softcap": case.softcap, "lens": case.len_kind,
         "work_per_step": (f"{decode_bytes(case):.4g} bytes" if is_decode(idx)
                           else f"{prefill_flops(case):.4g} flop")}
    if res is not None:
        c["l2"] = "flushed between steps (256 MB write)" if res["l2_flush"] else "inputs larger than L2"
    return c


if __name__ == "__main__":
    main()
