"""GPU parity: every entry point against the double-precision oracle, element by element.

Tolerances (max-abs error of the output, fp32 accumulation on the GPU): 1e-4 for fp32,
2e-2 for fp16/bf16 outputs.  present_key/present_value must be bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle_adapter import expected_present, problem
from scaled_dot_product_gb300 import sdpa
from scaled_dot_product_gb300.workloads import Case, as4d, make_case, workload

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from scaled_dot_product_gb300 import build
    build.build()
    torch.cuda.init()


def y_as_bnsh(case: Case, y_store: torch.Tensor) -> np.ndarray:
    return as4d(y_store.float().cpu(), case.q_layout, case.Nq).double().numpy()


def run_and_compare(case: Case, op: str = "fwd", rows=None):
    dcase = case.to("cuda")
    ws = sdpa.case_workspace(dcase, op)
    y, pk, pv = sdpa.run_case(dcase, op, workspace=ws)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    got = y_as_bnsh(case, y)
    pr = problem(case)
    tol = TOL[case.dtype]
    if rows is None:
        want = oracle.attention(pr)
        err = np.abs(got - want).max() if want.size else 0.0
    else:
        want, _ = oracle.attention_rows(pr, rows)
        sel = got[rows[:, 0], rows[:, 1], rows[:, 2]]
        err = np.abs(sel - want).max() if want.size else 0.0
    assert np.isfinite(got).all()
    assert err <= tol, f"{case.name} [{op}] max-abs error {err:.3e} > {tol}"
    if case.want_present:
        ek, ev = expected_present(case)
        assert torch.equal(pk.cpu().view(torch.int16 if case.dtype != torch.float32 else torch.int32),
                           ek.view(torch.int16 if case.dtype != torch.float32 else torch.int32))
        assert torch.equal(pv.cpu().view(torch.int16 if case.dtype != torch.float32 else torch.int32),
                           ev.view(torch.int16 if case.dtype != torch.float32 else torch.int32))
    return err, sdpa.sdpa_last_kernel_name()


# ----------------------------------------------------------------- the five workloads, small

@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5, 6])
def test_workload_small_fwd(idx):
    run_and_compare(workload(idx, small=True), "fwd")


def test_workload4_small_decode():
    err, name = run_and_compare(workload(4, small=True), "decode")
    assert name.startswith("decode_splitkv")


def test_workload1_exact_config():
    err, _ = run_and_compare(workload(1), "fwd")
    assert err <= 1e-4


# ----------------------------------------------------------------- randomized feature sweep

def _sweep_cases():
    rng = np.random.default_rng(2024)
    cases = []
    for n in range(24):
        dtype = [torch.float16, torch.bfloat16, torch.float32][n % 3]
        H = int(rng.choice([64, 128] if dtype != torch.float32 else [32, 64, 128]))
        Nkv = int(rng.choice([1, 2]))
        Nq = Nkv * int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        S = int(rng.choice([1, 2, 5, 17, 130, 257]))
        L = S if rng.random() < 0.6 else int(rng.integers(1, 300))
        P = 0 if rng.random() < 0.5 else int(rng.integers(1, 200))
        causal = str(rng.choice(["none", "upper_left", "lower_right"]))
        window = int(rng.integers(1, 64)) if (causal != "none" and rng.random() < 0.5) else -1
        T = P + L
        kw = dict(dtype=dtype, B=B, Nq=Nq, Nkv=Nkv, S=S, L=L, P=P, H=H, seed=5000 + n,
                  causal=causal, window=window, sink=bool(rng.random() < 0.4),
                  softcap=float(rng.choice([0.0, 0.0, 5.0, 30.0])),
                  q_layout=str(rng.choice(["bnsh", "bsnh"])),
                  kv_layout=str(rng.choice(["bnsh", "bsnh"])) if P == 0 else "bnsh",
                  want_present=bool(rng.random() < 0.4))
        m = rng.random()
        if m < 0.25:
            kw.update(add_mask="float", add_mask_shape=(B, 1, S, max(1, T - int(rng.integers(0, 3)))),
                      add_mask_range=(-2.0, 1.0))
        elif m < 0.45:
            kw.update(keep_kind="bool", keep_mask_shape=(1, Nq, S, T))
        elif m < 0.55:
            kw.update(keep_kind="filter", keep_mask_shape=(B, 1, 1, T))
        lk = rng.random()
        if lk < 0.2:
            kw.update(len_kind="nonpad", len_range=(1, T))
        elif lk < 0.35:
            kw.update(len_kind="keylen", len_range=(1, T))
        if rng.random() < 0.25:
            kw.update(qkv_bias="qkv" if P == 0 or rng.random() < 0.5 else "q")
        cases.append(make_case(f"sweep{n}", **kw))
    return cases


SWEEP = _sweep_cases()


@pytest.mark.parametrize("case", SWEEP, ids=[c.name for c in SWEEP])
def test_sweep_fwd(case):
    run_and_compare(case, "fwd")


@pytest.mark.parametrize("case", [c for c in SWEEP if c.S <= 16 and c.H == c.Hv and
                                  (c.dtype != torch.float32 or c.H in (32, 64, 128))],
                         ids=lambda c: c.name)
def test_sweep_decode(case):
    run_and_compare(case, "decode")


# ----------------------------------------------------------------- additive-mask row alignments

# Mask rows of Tm 16-bit columns start 4-, 8- or 16-byte aligned (Tm = 258, 260, 264) or only
# 2-byte aligned (Tm = 259); full mask tiles are staged through shared memory when the rows
# allow 4-byte copies, and the ragged last tile and 2-byte rows are read per thread.  S = 150
# leaves a partial query tile and partial 32-row groups.
@pytest.mark.parametrize("Tm", [258, 259, 260, 264])
@pytest.mark.parametrize("cap", ["none", "after", "before"])
def test_additive_mask_row_alignments(Tm, cap):
    for dtype, H in ((torch.float16, 64), (torch.bfloat16, 128)):
        c = make_case(f"addmask_t{Tm}_{cap}", dtype=dtype, B=2, Nq=4, Nkv=2, S=150, L=300, H=H, seed=40 + Tm,
                      add_mask="float", add_mask_shape=(2, 1, 150, Tm), add_mask_range=(-2.0, 1.0),
                      softcap=0.0 if cap == "none" else 5.0, softcap_before_bias=cap == "before",
                      causal="lower_right" if Tm % 2 else "none")
        err, name = run_and_compare(c, "fwd")
        assert name.startswith("prefill_tc"), name


# ----------------------------------------------------------------- edge cases

def test_no_keys_gives_zeros_and_sink_keeps_zero():
    for sink in (False, True):
        c = make_case("nokeys", dtype=torch.float16, B=1, Nq=2, S=3, L=0, H=64, sink=sink, seed=11)
        dcase = c.to("cuda")
        y, _, _ = sdpa.run_case(dcase, "fwd")
        torch.cuda.synchronize()
        assert torch.count_nonzero(y) == 0


def test_fully_excluded_rows_are_zero():
    c = make_case("allmasked", dtype=torch.bfloat16, B=1, Nq=2, S=40, L=40, H=64, seed=12,
                  keep_kind="bool", keep_mask_shape=(1, 1, 40, 40), keep_density=0.0)
    run_and_compare(c, "fwd")


def test_empty_batch_and_empty_query_write_present_only():
    c = make_case("emptyq", dtype=torch.float16, B=2, Nq=2, S=0, L=5, P=3, H=64, seed=13,
                  want_present=True)
    run_and_compare(c, "fwd")
    run_and_compare(c, "decode")


def test_head_size_256_and_distinct_value_width():
    run_and_compare(make_case("h256", dtype=torch.bfloat16, B=1, Nq=2, S=70, L=90, H=256, seed=14), "fwd")
    err, name = run_and_compare(make_case("hv", dtype=torch.float16, B=1, Nq=4, Nkv=2, S=33, L=70, H=64, Hv=128,
                                          seed=15, causal="lower_right"), "fwd")
    assert name.startswith("prefill_tc"), name


@pytest.mark.parametrize("kw", [
    dict(name="h64_hv128_gqa_causal_bf16", dtype=torch.bfloat16, H=64, Hv=128, Nkv=2, causal="upper_left",
         len_kind="nonpad", len_range=(150, 300)),
    dict(name="h128_hv64_window_sink_f16", dtype=torch.float16, H=128, Hv=64, causal="lower_right", window=70,
         sink=True),
    dict(name="h128_hv64_addmask_bf16", dtype=torch.bfloat16, H=128, Hv=64, add_mask="float",
         add_mask_shape=(2, 1, 260, 300)),
    dict(name="h64_hv128_bool_f16", dtype=torch.float16, H=64, Hv=128, keep_kind="bool",
         keep_mask_shape=(2, 4, 260, 300)),
    dict(name="h64_hv128_softcap_bf16", dtype=torch.bfloat16, H=64, Hv=128, causal="upper_left", softcap=20.0),
])
def test_distinct_value_width_tensor_core(kw):
    """Value head size different from the query/key one (64 / 128) on the tensor-core kernel."""
    kw = dict(kw)
    name = kw.pop("name")
    kw.setdefault("Nkv", 4)
    case = make_case(name, B=2, Nq=4, S=260, L=300, seed=80 + len(name), q_layout="bsnh", **kw)
    err, kernel = run_and_compare(case, "fwd")
    assert kernel.startswith("prefill_tc") and "_hv" in kernel, kernel


def test_softcap_after_bias_reading():
    c = make_case("capbias", dtype=torch.float32, B=1, Nq=2, S=9, L=11, H=32, seed=16, softcap=2.0,
                  add_mask="float", add_mask_range=(-3.0, 3.0))
    run_and_compare(c, "fwd")
    c.softcap_before_bias = True
    run_and_compare(c, "fwd")


def test_key_and_value_views_in_different_layouts():
    """K as (B, N, L, H) and V packed (B, L, N*Hv): the tensor-core kernel needs both views
    to walk their axes alike, so this takes the general path; the result must not change."""
    c = make_case("kv_mixed", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=150, L=150, H=64, seed=18,
                  causal="upper_left")
    dcase = c.to("cuda")
    q, k, v = dcase.views()
    v_packed = v.transpose(1, 2).contiguous().transpose(1, 2)       # same values, (s, n) swapped
    y = sdpa.sdpa_attn_fwd(q, k, v_packed, causal="upper_left")
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    err = np.abs(y.float().cpu().double().numpy() - oracle.attention(problem(c))).max()
    assert err <= TOL[c.dtype], err


def test_kv_concat_bit_exact_with_and_without_bias():
    for dtype in (torch.float16, torch.bfloat16, torch.float32):
        g = torch.Generator().manual_seed(17)
        past = torch.randn(2, 3, 37, 64, generator=g).to(dtype)
        cur = torch.randn(2, 3, 5, 64, generator=g).to(dtype)
        bias = (torch.randn(3 * 64, generator=g) * 0.02).to(dtype)
        for b in (None, bias):
            pres = torch.empty(2, 3, 42, 64, dtype=dtype, device="cuda")
            sdpa.sdpa_kv_concat(past.cuda(), cur.cuda(), pres, None if b is None else b.cuda())
            torch.cuda.synchronize()
            want = oracle.present(past, cur, b)
            iv = torch.int32 if dtype == torch.float32 else torch.int16
            assert torch.equal(pres.cpu().view(iv), want.view(iv)), (dtype, b is not None)


# ----------------------------------------------------------------- MultiHeadAttention projection bias

def test_mha_projection_bias_rank4_cross_attention():
    """The operator's single projection-bias input through sdpa_mha_fwd: with rank-4 key/value
    (the cross-attention workload) only the query segment applies, so non-zero key and value
    segments leave y bit-identical and equal to the oracle's; with rank-3 key/value every
    segment applies."""
    c = workload(5, small=True)
    N, H, Hv = c.Nq, c.H, c.Hv
    bias = c.proj_bias
    assert bias is not None and bias.numel() == 2 * N * H + N * Hv
    assert bias[N * H:].abs().max() > 0                       # the key / value segments are not zero
    zeroed = bias.clone()
    zeroed[N * H:] = 0
    d = c.to("cuda")
    am = d.add_mask
    y = sdpa.sdpa_mha_fwd(d.q, d.k, d.v, num_heads=N, projection_bias=bias.cuda(), add_mask=am,
                          mask_filter_value=c.mask_filter_value)
    y0 = sdpa.sdpa_mha_fwd(d.q, d.k, d.v, num_heads=N, projection_bias=zeroed.cuda(), add_mask=am,
                           mask_filter_value=c.mask_filter_value)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    pr = problem(c)
    pr.q_bias, pr.k_bias, pr.v_bias = oracle.mha_projection_bias(bias, N, H, Hv, kv_rank=4)
    want = oracle.attention(pr)
    err = np.abs(y_as_bnsh(c, y) - want).max()
    assert err <= TOL[c.dtype], err
    # the same problem with packed rank-3 key/value: the key and value segments apply
    k3 = d.k.permute(0, 2, 1, 3).reshape(c.B, c.L, N * H).contiguous()
    v3 = d.v.permute(0, 2, 1, 3).reshape(c.B, c.L, N * Hv).contiguous()
    y3 = sdpa.sdpa_mha_fwd(d.q, k3, v3, num_heads=N, projection_bias=bias.cuda(), add_mask=am,
                           mask_filter_value=c.mask_filter_value)
    torch.cuda.synchronize()
    pr.q_bias, pr.k_bias, pr.v_bias = oracle.mha_projection_bias(bias, N, H, Hv, kv_rank=3)
    err3 = np.abs(y_as_bnsh(c, y3) - oracle.attention(pr)).max()
    assert err3 <= TOL[c.dtype], err3


# ----------------------------------------------------------------- full-size workloads, every row

@pytest.mark.slow
@pytest.mark.parametrize("idx,op", [(2, "fwd"), (3, "fwd"), (4, "decode"), (4, "fwd"), (5, "fwd"), (6, "fwd")])
def test_workload_full_size(idx, op):
    """Every output element of the full-size workloads (the configuration bench.py times)
    against the oracle, and present bit-exact; the oracle takes seconds per workload on the
    host's cores."""
    run_and_compare(workload(idx), op)


# ----------------------------------------------------------------- bf16 softcap, fixed maximum

@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("softcap,q_gain,sink", [
    (30.0, 1.0, False),    # cubic tanh throughout
    (30.0, 1.0, True),     # sink below the cap
    (3.0, 1.0, True),      # arguments beyond the cubic's range: tanh on the special-function unit
    (40.0, 12.0, False),   # logits near +-c: weights down to 2^(-2 c log2 e)
    (8.0, 2.0, "big"),     # sink logit above the cap: it becomes the fixed maximum
    (55.0, 3.0, False),    # cap above 40: the running-maximum path
])
def test_bf16_softcap_fixed_maximum(H, softcap, q_gain, sink):
    """Softcap bounds every logit by +-c, so the bf16 kernel uses c (or a larger sink logit)
    as the softmax maximum instead of a running one; results must not change."""
    c = make_case(f"capfix_h{H}_c{softcap:g}", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=300, L=300, H=H,
                  seed=40 + H, causal="upper_left", softcap=softcap, sink=bool(sink),
                  len_kind="nonpad", len_range=(120, 300), q_layout="bsnh", kv_layout="bsnh")
    if q_gain != 1.0:
        c.q = (c.q.float() * q_gain).to(torch.bfloat16)
    if sink == "big":
        c.head_sink = (torch.arange(c.Nq, dtype=torch.float32) * 3.0 + softcap + 2.0).to(torch.bfloat16)
    err, name = run_and_compare(c, "fwd")
    assert name.startswith("prefill_tc"), name


# ----------------------------------------------------------------- keep masks on the tensor-core path

@pytest.mark.parametrize("kw", [
    dict(name="bool_ul_bf16_h128", dtype=torch.bfloat16, H=128, causal="upper_left", keep_kind="bool",
         keep_mask_shape=(2, 1, 200, 320)),
    dict(name="bool_short_f16_h64", dtype=torch.float16, H=64, keep_kind="bool",
         keep_mask_shape=(1, 4, 200, 301)),                 # rows not 16-byte aligned, shorter than T
    dict(name="filter_lr_f16_h128", dtype=torch.float16, H=128, causal="lower_right", keep_kind="filter",
         keep_mask_shape=(2, 1, 200, 320)),
    dict(name="filter_keylen_bf16_h64", dtype=torch.bfloat16, H=64, keep_kind="filter",
         keep_mask_shape=(2, 1, 1, 320), len_kind="keylen", len_range=(5, 320)),
    dict(name="keylen_only_f16_h128", dtype=torch.float16, H=128, causal="lower_right", len_kind="keylen",
         len_range=(1, 320), sink=True),
    dict(name="bool_window_gqa_bf16_h64", dtype=torch.bfloat16, H=64, Nkv=2, causal="lower_right", window=90,
         keep_kind="bool", keep_mask_shape=(2, 4, 200, 320)),
])
def test_keep_masks_tensor_core_path(kw):
    kw = dict(kw)
    name = kw.pop("name")
    kw.setdefault("Nkv", 4)
    case = make_case(name, B=2, Nq=4, S=200, L=320, seed=60 + len(name), keep_density=0.85, **kw)
    err, kernel = run_and_compare(case, "fwd")
    assert kernel.startswith("prefill_tc"), kernel


def test_keep_mask_excluding_whole_rows_gives_zeros():
    c = make_case("bool_allfalse", dtype=torch.bfloat16, B=1, Nq=2, S=150, L=150, H=64, seed=71,
                  keep_kind="bool", keep_mask_shape=(1, 1, 150, 150), keep_density=0.0)
    run_and_compare(c, "fwd")


# ----------------------------------------------------------------- many launches, barrier phases

@pytest.mark.parametrize("kw", [
    # P aliasing S (Hv = 128): the unit's last P.V and the next unit's first S complete back to
    # back; the epilogue must wait on its own barrier, not on a second phase of the score one
    dict(name="stress_keep_f16_h128", dtype=torch.float16, B=2, Nq=16, Nkv=16, S=1024, L=1024, H=128,
         q_layout="bsnh", kv_layout="bsnh", causal="lower_right", keep_kind="filter",
         keep_mask_shape=(2, 1, 1024, 1024), seed=91),
    dict(name="stress_capfix_bf16_h128", dtype=torch.bfloat16, B=2, Nq=16, Nkv=4, S=1024, L=1024, H=128,
         causal="upper_left", softcap=30.0, len_kind="nonpad", len_range=(600, 1024), seed=92),
    dict(name="stress_plain_bf16_h64", dtype=torch.bfloat16, B=1, Nq=32, Nkv=4, S=2048, L=2048, H=64,
         causal="lower_right", window=512, sink=True, seed=93),
])
def test_many_launches_keep_every_barrier_phase(kw):
    """Hundreds of back-to-back launches of the persistent kernel (several units per CTA):
    every one completes without a bounded wait expiring, and the last result matches the
    oracle on sampled rows."""
    c = make_case(**kw)
    d = c.to("cuda")
    ws = sdpa.case_workspace(d, "fwd")
    outs = sdpa.case_outputs(d)
    for _ in range(400):
        sdpa.run_case(d, "fwd", outputs=outs, workspace=ws)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK, sdpa.sdpa_last_error()
    assert sdpa.sdpa_last_kernel_name().startswith("prefill_tc"), sdpa.sdpa_last_kernel_name()
    got = y_as_bnsh(c, outs[0])
    rng = np.random.default_rng(7)
    rows = np.stack([rng.integers(0, c.B, 64), rng.integers(0, c.Nq, 64), rng.integers(0, c.S, 64)], 1)
    want, _ = oracle.attention_rows(problem(c), rows)
    err = np.abs(got[rows[:, 0], rows[:, 1], rows[:, 2]] - want).max()
    assert err <= TOL[c.dtype], f"{c.name}: max-abs error {err:.3e}"
