"""GPU parity of the rotary embedding (class RotaryEmbedding) against the oracle.

Standalone: sdpa_rotary over rank-3 and rank-4 inputs, rank-2 caches with position ids and
rank-3 per-token caches, both pair layouts, partial rotary_dim.  Inside attention:
GroupQueryAttention's rotation of Q and the new K rows at absolute positions, on the
tensor-core, SIMT and decode paths, with present holding the rotated keys.

Bounds.  The oracle rotates in float64 and rounds once to the element type; the kernel
computes x1*c - x2*s in float32 and rounds that to the element type.  For 16-bit inputs
both products are exact in float32, so the two differ at most by the float32 rounding of
the sum before the final rounding; for float32 inputs the rounded product x2*s adds up to
half an ulp of |x2 s|.  Each rotated element must therefore lie within
2^-m |want| + 2^-23 (|x1| + |x2|) of the oracle (m = stored mantissa bits: one ulp of the
element type plus the float32 term); copied channels must be bit-equal.  Attention outputs
keep the usual 1e-4 (fp32) / 2e-2 (fp16, bf16) max-abs bounds.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_adapter import expected_present, problem
from scaled_dot_product_gb300 import sdpa
from scaled_dot_product_gb300.workloads import as4d, make_case, make_rotary_inputs

pytestmark = pytest.mark.gpu

MANT = {torch.float32: 23, torch.float16: 10, torch.bfloat16: 7}
TOL = {torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from scaled_dot_product_gb300 import build
    build.build()
    torch.cuda.init()


def _partner_mag(x: np.ndarray, R: int, interleaved: bool) -> np.ndarray:
    """|x_i| + |x_partner(i)| on the rotated channels, 0 on the copied ones."""
    a = np.abs(x)
    out = np.zeros_like(a)
    h = R // 2
    if interleaved:
        s = a[..., 0:R:2] + a[..., 1:R:2]
        out[..., 0:R:2] = s
        out[..., 1:R:2] = s
    else:
        s = a[..., :h] + a[..., h:R]
        out[..., :h] = s
        out[..., h:R] = s
    return out


def check_rotated(got: torch.Tensor, x: torch.Tensor, want: np.ndarray, R: int, interleaved: bool):
    """got, x: (B, N, S, D) views (dtype); want: oracle float64 (B, N, S, D)."""
    g = got.float().cpu().double().numpy()
    xs = x.float().cpu().double().numpy()
    m = MANT[got.dtype]
    bound = 2.0 ** -m * np.abs(want) + 2.0 ** -23 * _partner_mag(xs, R, interleaved)
    err = np.abs(g - want)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{bad.shape[0]} elements outside the bound, first {bad[0]}: got " \
                          f"{g[tuple(bad[0])]} want {want[tuple(bad[0])]}"
    if R < x.shape[-1]:
        assert torch.equal(got[..., R:].cpu(), x[..., R:].cpu())


# ------------------------------------------------------------------------------ standalone

STANDALONE = [
    dict(dtype=torch.float32, layout="bnsh", interleaved=False, rotary_dim=0, cache="ids"),
    dict(dtype=torch.float16, layout="bsnh", interleaved=True, rotary_dim=0, cache="ids"),
    dict(dtype=torch.bfloat16, layout="bnsh", interleaved=False, rotary_dim=32, cache="per_token"),
    dict(dtype=torch.bfloat16, layout="bsnh", interleaved=True, rotary_dim=48, cache="ids"),
    dict(dtype=torch.float16, layout="bnsh", interleaved=False, rotary_dim=16, cache="per_token", D=128),
    dict(dtype=torch.float32, layout="bsnh", interleaved=True, rotary_dim=8, cache="ids", D=32),
    # R/2 not a multiple of a 16-byte vector: the scalar kernel
    dict(dtype=torch.float16, layout="bnsh", interleaved=False, rotary_dim=12, cache="ids"),
    dict(dtype=torch.bfloat16, layout="bsnh", interleaved=True, rotary_dim=6, cache="per_token"),
]


@pytest.mark.parametrize("cfg", STANDALONE, ids=[f"{c['dtype']}-{c['layout']}-i{int(c['interleaved'])}-"
                                                 f"r{c['rotary_dim']}-{c['cache']}" for c in STANDALONE])
def test_standalone_rotary_matches_oracle(cfg):
    cfg = dict(cfg)
    D = cfg.pop("D", 64)
    ri = make_rotary_inputs(B=3, N=5, S=37, D=D, seed=11, **cfg)
    d = ri.to("cuda")
    y = sdpa.sdpa_rotary(d.x, d.cos, d.sin, d.position_ids, rotary_dim=ri.rotary_dim,
                         interleaved=ri.interleaved, num_heads=ri.N)
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    assert sdpa.sdpa_last_kernel_name() == "rotary"
    x4 = as4d(ri.x, ri.layout, ri.N)
    want = oracle.rotary(x4, ri.cos, ri.sin, ri.position_ids, ri.rotary_dim, ri.interleaved)
    check_rotated(as4d(y.cpu(), ri.layout, ri.N), x4, want, ri.rotary_dim or D, ri.interleaved)


def test_standalone_rotary_in_place_and_empty():
    ri = make_rotary_inputs(B=2, N=4, S=300, D=128, dtype=torch.bfloat16, seed=3)
    d = ri.to("cuda")
    x0 = d.x.clone()
    sdpa.sdpa_rotary(d.x, d.cos, d.sin, d.position_ids, y=d.x)       # y is x
    want = oracle.rotary(ri.x, ri.cos, ri.sin, ri.position_ids)
    check_rotated(d.x, x0, want, 128, False)
    e = torch.empty(0, 4, 5, 128, dtype=torch.bfloat16, device="cuda")
    sdpa.sdpa_rotary(e, d.cos, d.sin, torch.zeros(0, 5, dtype=torch.int64, device="cuda"))
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK


def test_vector_and_scalar_kernels_agree_bit_for_bit():
    """A view whose rows start off a 16-byte boundary takes the scalar kernel; the same
    values in an aligned tensor take the vector kernel.  Both round x1 c - x2 s once."""
    for dtype in (torch.bfloat16, torch.float16, torch.float32):
        for inter in (False, True):
            ri = make_rotary_inputs(B=2, N=3, S=45, D=64, dtype=dtype, interleaved=inter, seed=21)
            d = ri.to("cuda")
            store = torch.zeros(2, 3, 45, 66, dtype=dtype, device="cuda")
            xm = store[..., 1:65]                                       # misaligned rows
            xm.copy_(d.x)
            y_vec = sdpa.sdpa_rotary(d.x, d.cos, d.sin, d.position_ids, interleaved=inter)
            y_sca = sdpa.sdpa_rotary(xm, d.cos, d.sin, d.position_ids, interleaved=inter)
            assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
            iv = torch.int32 if dtype == torch.float32 else torch.int16
            assert torch.equal(y_vec.view(iv), y_sca.contiguous().view(iv)), (dtype, inter)
            check_rotated(y_sca, ri.x, oracle.rotary(ri.x, ri.cos, ri.sin, ri.position_ids, 0, inter), 64, inter)


def test_position_outside_the_cache_is_reported_and_the_context_survives():
    ri = make_rotary_inputs(B=1, N=2, S=8, D=64, dtype=torch.float16, seed=5, max_pos=16)
    d = ri.to("cuda")
    bad = d.position_ids.clone()
    bad[0, 3] = 16                                                   # one past the last row
    sdpa.sdpa_rotary(d.x, d.cos, d.sin, bad)
    assert sdpa.sdpa_query_status() == sdpa.SDPA_ERR_INVALID
    y = sdpa.sdpa_rotary(d.x, d.cos, d.sin, d.position_ids)
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    check_rotated(y, ri.x, oracle.rotary(ri.x, ri.cos, ri.sin, ri.position_ids), 64, False)


# ------------------------------------------------------------------------------ inside attention

def _rot_cases():
    return [
        # tensor-core path (H=128), GQA, seqlens_k = total - 1, causal lower-right
        make_case("rope_gqa_prefill_bf16_h128", dtype=torch.bfloat16, B=2, Nq=8, Nkv=2, S=300, H=128,
                  q_layout="bsnh", kv_layout="bsnh", causal="lower_right", rotary="half", seed=41,
                  want_present=True),
        # tensor-core path (H=64), window + sink, interleaved partial rotation
        make_case("rope_gqa_window_bf16_h64_r32", dtype=torch.bfloat16, B=1, Nq=8, Nkv=2, S=260, H=64,
                  causal="lower_right", window=70, sink=True, rotary="interleaved", rotary_dim=32,
                  seed=42),
        # past rows + present (materialised K), f16 tensor-core path
        make_case("rope_past_f16_h64", dtype=torch.float16, B=2, Nq=4, Nkv=4, S=130, P=90, H=64,
                  causal="lower_right", rotary="half", seed=43, want_present=True),
        # SIMT path (fp32), cross lengths S != L, partial interleaved rotation
        make_case("rope_f32_cross", dtype=torch.float32, B=1, Nq=4, Nkv=2, S=20, L=27, P=7, H=32,
                  causal="lower_right", rotary="interleaved", rotary_dim=16, seed=44, want_present=True),
    ]


def _seqlens(case):
    case.lens = torch.full((case.B,), case.T - 1, dtype=torch.int32)
    case.len_kind = "seqlens_k"
    return case


def _run(case, op):
    dcase = case.to("cuda")
    ws = sdpa.case_workspace(dcase, op)
    y, pk, pv = sdpa.run_case(dcase, op, workspace=ws)
    torch.cuda.synchronize()
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
    got = as4d(y.float().cpu(), case.q_layout, case.Nq).double().numpy()
    want = oracle.attention(problem(case))
    err = np.abs(got - want).max() if want.size else 0.0
    assert err <= TOL[case.dtype], f"{case.name} [{op}] max-abs error {err:.3e}"
    if case.want_present:
        ek, ev = expected_present(case)
        # the rotated rows within the bound of check_rotated, past rows and values bit-exact
        assert torch.equal(pv.cpu(), ev)
        assert torch.equal(pk[:, :, :case.P].cpu(), ek[:, :, :case.P])
        _, k, _ = case.views()
        qpos, kpos = oracle.gqa_rotary_positions(case.B, case.S, case.L, case.T,
                                                 case.lens if case.len_kind == "seqlens_k" else None)
        wk = oracle.rotary(k, case.rotary_cos, case.rotary_sin, kpos, case.rotary_dim,
                           case.rotary_interleaved)
        check_rotated(pk[:, :, case.P:], k, wk, case.rotary_dim or case.H, case.rotary_interleaved)
    return sdpa.sdpa_last_kernel_name()


@pytest.mark.parametrize("i", range(4))
def test_attention_with_rotary_fwd(i):
    case = _rot_cases()[i]
    if i in (0, 1):
        case = _seqlens(case)
    name = _run(case, "fwd")
    if case.dtype != torch.float32:
        assert name.startswith("prefill_tc"), name


def test_attention_with_rotary_decode():
    case = make_case("rope_decode_f16_h128", dtype=torch.float16, B=4, Nq=8, Nkv=2, S=1, L=1, P=700,
                     H=128, q_layout="bsnh", kv_layout="bsnh", rotary="half", seed=45, want_present=True,
                     rotary_max_pos=1024)
    case.lens = torch.tensor([700, 350, 699, 10], dtype=torch.int32)    # seqlens_k per batch
    case.len_kind = "seqlens_k"
    name = _run(case, "decode")
    assert name.startswith("decode_splitkv")


def test_rotary_without_enough_cache_rows_is_reported():
    case = make_case("rope_short_cache", dtype=torch.bfloat16, B=1, Nq=2, Nkv=2, S=40, H=64,
                     causal="lower_right", rotary="half", rotary_max_pos=30, seed=46)
    dcase = case.to("cuda")
    sdpa.run_case(dcase, "fwd", workspace=sdpa.case_workspace(dcase, "fwd"))
    assert sdpa.sdpa_query_status() == sdpa.SDPA_ERR_INVALID
    assert sdpa.sdpa_query_status() == sdpa.SDPA_OK                    # the word was cleared
