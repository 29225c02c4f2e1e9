"""GPU parity of the backward (sdpa_attn_bwd) against the double-precision oracle's
backward (the GroupQueryAttention gradient graph), element by element on dQ, dK and dV."""
import numpy as np
import pytest
import torch

import oracle
from oracle_adapter import problem
from scaled_dot_product_gb300 import sdpa
from scaled_dot_product_gb300.workloads import as4d, draw_dy, make_case, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from scaled_dot_product_gb300 import build
    build.build()
    torch.cuda.init()


def run_bwd(case, dy):
    d = case.to("cuda")
    q, k, v = d.views()
    dy4 = as4d(dy.to("cuda"), case.q_layout, case.Nq)
    kw = sdpa.case_kwargs(d)
    dq, dk, dv = sdpa.sdpa_attn_bwd(q, k, v, dy4, **kw)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    assert sdpa.sdpa_last_kernel_name().startswith("bwd_tc")
    return dq.float().cpu().double().numpy(), dk.float().cpu().double().numpy(), dv.float().cpu().double().numpy()


def compare(case, dy, report=None):
    got = run_bwd(case, dy)
    want = oracle.backward(problem(case), as4d(dy, case.q_layout, case.Nq))
    stats = []
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        assert g.shape == w.shape, (name, g.shape, w.shape)
        assert np.isfinite(g).all(), name
        err = np.abs(g - w)
        scale = max(np.abs(w).max(), 1e-30)
        stats.append((name, float(err.max()), float(scale)))
        # rounding of the output (one ulp of the dtype at |want|) plus the 16-bit P / dS
        # operands of the products, bounded against the tensor's largest entry
        ulp = 2.0 ** (-8 if case.dtype == torch.bfloat16 else -10)
        bound = ulp * np.abs(w) + 2.0 * ulp * scale + 1e-6
        bad = err > bound
        assert not bad.any(), f"{case.name} {name}: {int(bad.sum())} entries off, max err {err.max():.3e}, max |want| {scale:.3e}"
    if report is not None:
        report.append((case.name, stats))
    return stats


CASES = [
    dict(name="plain_bf16_h64", dtype=torch.bfloat16, B=1, Nq=2, S=130, L=150, H=64),
    dict(name="plain_f16_h128", dtype=torch.float16, B=2, Nq=2, S=257, L=257, H=128),
    dict(name="gqa4_causal_ul_bf16_h128", dtype=torch.bfloat16, B=2, Nq=8, Nkv=2, S=300, L=300, H=128,
         causal="upper_left", q_layout="bsnh", kv_layout="bsnh"),
    dict(name="gqa2_lr_window_sink_f16_h64", dtype=torch.float16, B=1, Nq=4, Nkv=2, S=200, L=333, H=64,
         causal="lower_right", window=70, sink=True),
    dict(name="nonpad_causal_bf16_h64", dtype=torch.bfloat16, B=3, Nq=2, Nkv=1, S=260, L=260, H=64,
         causal="upper_left", len_kind="nonpad", len_range=(1, 260)),
    dict(name="seqlens_k_window_sink_bf16_h128", dtype=torch.bfloat16, B=2, Nq=4, Nkv=1, S=190, L=190, H=128,
         causal="lower_right", window=64, sink=True, len_kind="seqlens_k", len_range=(100, 189)),
    dict(name="s_shorter_than_t_bf16_h64", dtype=torch.bfloat16, B=1, Nq=2, S=17, L=400, H=64,
         causal="lower_right"),
]


@pytest.mark.parametrize("kw", CASES, ids=[c["name"] for c in CASES])
def test_backward_matches_oracle(kw):
    kw = dict(kw)
    name = kw.pop("name")
    case = make_case(name, seed=900 + len(name), **kw)
    dy = draw_dy(case, seed=77 + len(name))
    compare(case, dy)


def test_backward_large_sink_and_empty_key_rows():
    """A sink far above every score takes almost all the mass (gradients near zero); keys
    beyond nonpad_kv_seqlen get exactly zero dK / dV."""
    case = make_case("bigsink", dtype=torch.bfloat16, B=2, Nq=2, S=140, L=140, H=64, causal="upper_left",
                     sink=True, len_kind="nonpad", len_range=(50, 90), seed=31)
    case.head_sink = torch.full((2,), 12.0, dtype=torch.bfloat16)
    dy = draw_dy(case, seed=32)
    compare(case, dy)
    _, dk, dv = run_bwd(case, dy)
    lens = case.lens.numpy()
    for b in range(case.B):
        assert np.all(dk[b, :, lens[b]:] == 0) and np.all(dv[b, :, lens[b]:] == 0)


def test_backward_workload3_small():
    """The GroupQueryAttention workload (window, sink, seqlens_k), small shape."""
    case = workload(3, small=True)
    compare(case, draw_dy(case, seed=303))


@pytest.mark.slow
def test_backward_full_size_gqa_key_gradient_sums_to_zero_without_sink():
    """At the full GroupQueryAttention workload size (S = 4096, 64 / 8 heads, window 1024,
    seqlens_k) but without the sink, every row of dS sums to zero (softmax backward), so
    sum_j dK_j = sum_i (sum_j dS_ij) Q_i = 0 for every (batch, kv head)."""
    case = workload(3)
    case.head_sink = None
    d = case.to("cuda")
    q, k, v = d.views()
    dy = as4d(draw_dy(case, seed=404).to("cuda"), case.q_layout, case.Nq)
    dq, dk, dv = sdpa.sdpa_attn_bwd(q, k, v, dy, **sdpa.case_kwargs(d))
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    dkf = dk.float()
    col = dkf.sum(dim=2)                       # (B, Nkv, H)
    mag = dkf.abs().sum(dim=2)
    assert torch.isfinite(dkf).all()
    assert (col.abs() <= 0.02 * mag + 1e-3).all(), float((col.abs() / (mag + 1e-6)).max())
    assert dq.abs().sum() > 0 and dv.abs().sum() > 0


MASK_CASES = [
    dict(name="addmask_bf16_h64", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=150, L=210, H=64,
         add_mask="float", add_mask_shape=(2, 1, 150, 210), add_mask_range=(-2.0, 1.0), causal="lower_right"),
    dict(name="addmask_short_f16_h128", dtype=torch.float16, B=1, Nq=2, S=130, L=200, H=128,
         add_mask="float", add_mask_shape=(1, 2, 130, 190), add_mask_range=(-1.0, 0.5)),
    dict(name="bool_mask_bf16_h64", dtype=torch.bfloat16, B=2, Nq=2, S=140, L=140, H=64,
         keep_kind="bool", keep_mask_shape=(2, 1, 140, 140), causal="upper_left"),
    dict(name="filter_keylen_f16_h64", dtype=torch.float16, B=2, Nq=4, Nkv=1, S=100, L=260, H=64,
         keep_kind="filter", keep_mask_shape=(2, 1, 1, 260), len_kind="keylen", len_range=(30, 260), sink=True),
    dict(name="keylen_bf16_h128", dtype=torch.bfloat16, B=2, Nq=2, S=200, L=200, H=128, causal="lower_right",
         len_kind="keylen", len_range=(50, 200)),
]


@pytest.mark.parametrize("kw", MASK_CASES, ids=[c["name"] for c in MASK_CASES])
def test_backward_with_masks_matches_oracle(kw):
    kw = dict(kw)
    name = kw.pop("name")
    case = make_case(name, seed=1300 + len(name), keep_density=0.8, **kw)
    compare(case, draw_dy(case, seed=1400 + len(name)))


PAST_BIAS_CASES = [
    dict(name="past_rows_causal_bf16_h64", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=150, L=150, P=90, H=64,
         causal="lower_right"),
    dict(name="past_rows_seqlens_k_f16_h128", dtype=torch.float16, B=2, Nq=2, Nkv=1, S=70, L=70, P=200, H=128,
         causal="lower_right", len_kind="seqlens_k", len_range=(150, 269), sink=True),
    dict(name="mha_qkv_bias_bf16_h64", dtype=torch.bfloat16, B=2, Nq=4, S=140, L=180, H=64, q_layout="bsnh",
         kv_layout="bsnh", qkv_bias="qkv", proj_bias_std=0.3),
    dict(name="mha_q_bias_past_f16_h64", dtype=torch.float16, B=1, Nq=2, S=130, L=130, P=60, H=64, qkv_bias="q",
         proj_bias_std=0.3, causal="lower_right"),
]


@pytest.mark.parametrize("kw", PAST_BIAS_CASES, ids=[c["name"] for c in PAST_BIAS_CASES])
def test_backward_with_past_rows_and_biases_matches_oracle(kw):
    """dK / dV cover the past rows followed by the new ones; the biases shift the rows the
    scores see, so the gradients are taken at the biased rows."""
    kw = dict(kw)
    name = kw.pop("name")
    case = make_case(name, seed=1500 + len(name), **kw)
    compare(case, draw_dy(case, seed=1600 + len(name)))
