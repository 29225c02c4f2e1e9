"""GPU parity of the auxiliary qk output (class Attention, qk_matmul_output_mode 0-3)
against the oracle, on the tensor-core kernel and on the general kernel.

Bound: the output is FLOAT whatever the input type.  Products of 16-bit inputs are exact
in fp32 and accumulate in fp32 (tensor cores or FMA), so a finite entry must lie within
1e-4 + 1e-6 |want| of the oracle (the relative term covers mask_filter_value offsets of
order 1e4, whose fp32 spacing is about 1e-3).  Excluded entries must match exactly: -inf
in stages 1 and 2, 0 in stage 3.  The attention output y keeps its own bound.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_adapter import problem
from scaled_dot_product_gb300 import sdpa
from scaled_dot_product_gb300.workloads import as4d, make_case

pytestmark = pytest.mark.gpu

TOL_Y = {torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from scaled_dot_product_gb300 import build
    build.build()
    torch.cuda.init()


def run_qk(case, mode, want_kernel=None):
    d = case.to("cuda")
    y_store, y4, pk, pv = sdpa.case_outputs(d)
    out = torch.full((case.B, case.Nq, case.S, case.T), float("nan"), dtype=torch.float32, device="cuda")
    q, k, v = d.views()
    kw = sdpa.case_kwargs(d, pk, pv)
    sdpa.sdpa_attn_fwd(q, k, v, y=y4, qk_out=out, qk_mode=mode, **kw)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    name = sdpa.sdpa_last_kernel_name()
    if want_kernel:
        assert want_kernel in name, name
    pr = problem(case)
    got = out.cpu().double().numpy()
    want = oracle.qk(pr, mode)
    inf_w, inf_g = np.isinf(want), np.isinf(got)
    assert not np.isnan(got).any(), "unwritten entries"
    np.testing.assert_array_equal(inf_g, inf_w)
    np.testing.assert_array_equal(got[inf_w], want[inf_w])
    fin = ~inf_w
    err = np.abs(got[fin] - want[fin]) - (1e-4 + 1e-6 * np.abs(want[fin]))
    assert err.size == 0 or err.max() <= 0, f"mode {mode}: worst excess {err.max():.3e}"
    if mode == 3:
        np.testing.assert_array_equal(got[want == 0.0], 0.0)
    ygot = as4d(y_store.float().cpu(), case.q_layout, case.Nq).double().numpy()
    assert np.abs(ygot - oracle.attention(pr)).max() <= TOL_Y[case.dtype]
    return name


CASES = {
    # tensor-core kernel, H=128, GQA, causal, softcap, nonpad lengths, ragged S and T
    "tc_bf16_h128_causal_softcap": lambda: make_case(
        "qk_a", dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=300, H=128, q_layout="bsnh", kv_layout="bsnh",
        causal="upper_left", softcap=3.0, len_kind="nonpad", len_range=(150, 300), seed=91),
    # tensor-core kernel, H=64, short additive mask (-inf padding), window, sink, seqlens_k
    "tc_f16_h64_mask_window_sink": lambda: _seqlens(make_case(
        "qk_b", dtype=torch.float16, B=1, Nq=4, Nkv=1, S=200, H=64, causal="lower_right", window=50,
        sink=True, add_mask="float", add_mask_shape=(1, 4, 200, 180), add_mask_range=(-2.0, 1.0), seed=92)),
    # tensor-core kernel reading K from present (past rows), f16 H=128
    "tc_f16_h128_past_present": lambda: make_case(
        "qk_c", dtype=torch.float16, B=2, Nq=2, Nkv=2, S=140, P=60, H=128, causal="lower_right",
        want_present=True, seed=93),
}
GENERAL = {
    # general kernel: fp32
    "simt_f32_past_bias_filter": lambda: make_case(
        "qk_d", dtype=torch.float32, B=1, Nq=4, Nkv=4, S=20, L=23, P=9, H=32, seed=94, qkv_bias="qkv",
        keep_kind="filter", keep_mask_shape=(1, 1, 20, 32), mask_filter_value=-10000.0, softcap=2.0),
    # general kernel: past rows without a present output (no single K view)
    "simt_bf16_past_no_present": lambda: make_case(
        "qk_e", dtype=torch.bfloat16, B=2, Nq=2, Nkv=1, S=33, L=40, P=17, H=64, causal="lower_right",
        seed=95),
    # general kernel: T not a multiple of 4 (the fp32 output rows are not 16-byte aligned)
    "simt_bf16_ragged_T": lambda: make_case(
        "qk_f", dtype=torch.bfloat16, B=1, Nq=2, Nkv=2, S=70, L=301, H=64, seed=96,
        keep_kind="bool", keep_mask_shape=(1, 2, 70, 301), keep_density=0.7),
}


def _seqlens(case):
    case.lens = torch.full((case.B,), case.T - 1, dtype=torch.int32)
    case.len_kind = "seqlens_k"
    return case


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("name", sorted(CASES))
def test_qk_tensor_core(name, mode):
    run_qk(CASES[name](), mode, want_kernel="qk_tc")


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("name", sorted(GENERAL))
def test_qk_general(name, mode):
    run_qk(GENERAL[name](), mode, want_kernel="qk_simt")


def test_qk_rows_with_nothing_admitted():
    c = make_case("qk_g", dtype=torch.bfloat16, B=1, Nq=2, Nkv=2, S=130, L=132, H=128, seed=97,
                  keep_kind="bool", keep_mask_shape=(1, 1, 130, 132), keep_density=0.0)
    for mode in (1, 3):
        run_qk(c, mode, want_kernel="qk_tc")
