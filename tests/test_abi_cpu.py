"""C-ABI checks that need no GPU: the library loads, exports every symbol include/sdpa.h
declares, and rejects every invalid argument with its documented code before any launch."""
import ctypes
import os
import re

import pytest
import torch

from scaled_dot_product_gb300 import build as sdpa_build
from scaled_dot_product_gb300 import sdpa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module", autouse=True)
def library():
    sdpa_build.build()
    return sdpa.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SDPA_API\s+[\w\s\*]+?\b(sdpa_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 9
    lib = sdpa.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(sdpa.EXPORTED)


def test_version_and_empty_error():
    assert "sm_103a" in sdpa.sdpa_version()


def base(dtype=torch.bfloat16, B=2, Nq=4, Nkv=2, S=8, L=8, P=0, H=64, Hv=64, **kw):
    q = torch.zeros(B, Nq, S, H, dtype=dtype)
    k = torch.zeros(B, Nkv, L, H, dtype=dtype)
    v = torch.zeros(B, Nkv, L, Hv, dtype=dtype)
    y = torch.zeros(B, Nq, S, Hv, dtype=dtype)
    if P:
        kw.setdefault("past_k", torch.zeros(B, Nkv, P, H, dtype=dtype))
        kw.setdefault("past_v", torch.zeros(B, Nkv, P, Hv, dtype=dtype))
    return sdpa.make_params(q, k, v, y=y, **kw)


def code(params_keep, op=sdpa.SDPA_OP_FWD):
    params, _keep = params_keep
    return sdpa.sdpa_validate(params, op)


def test_valid_problems_validate():
    assert code(base()) == sdpa.SDPA_OK
    assert code(base(P=5)) == sdpa.SDPA_OK
    assert code(base(causal="lower_right", window=3)) == sdpa.SDPA_OK
    assert code(base(S=1, L=1, P=7, H=128, Hv=128, dtype=torch.float16), sdpa.SDPA_OP_DECODE) == sdpa.SDPA_OK
    assert code(base(dtype=torch.float32, H=8, Hv=8)) == sdpa.SDPA_OK


@pytest.mark.parametrize("window", [0, -2, -100, 2 ** 31])
def test_window_values_outside_the_contract_are_invalid(window):
    assert code(base(causal="upper_left", window=window)) == sdpa.SDPA_ERR_INVALID


def test_window_without_causal_is_invalid():
    assert code(base(window=16)) == sdpa.SDPA_ERR_INVALID


def test_group_mismatch_is_a_shape_error():
    assert code(base(Nq=3, Nkv=2)) == sdpa.SDPA_ERR_SHAPE


@pytest.mark.parametrize("H", [12, 264])
def test_unsupported_head_sizes(H):
    assert code(base(H=H, Hv=64)) == sdpa.SDPA_ERR_UNSUPPORTED


def test_struct_size_and_null_params():
    p, keep = base()
    p.struct_size = 4
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_INVALID
    assert sdpa.lib().sdpa_validate(None, 0) == sdpa.SDPA_ERR_NULL
    assert sdpa.lib().sdpa_attn_fwd(None, None, 0, None) == sdpa.SDPA_ERR_NULL


def test_bad_enums_and_non_finite_attributes():
    for kw in (dict(causal=7), dict(keep_kind=9, keep_mask=torch.ones(1, 1, 8, 8, dtype=torch.uint8)),
               dict(softcap=float("nan")), dict(softcap=float("inf")), dict(scale=float("nan")),
               dict(mask_filter_value=float("-inf"))):
        assert code(base(**kw)) == sdpa.SDPA_ERR_INVALID, kw
    p, keep = base()
    p.len_kind = 2          # lengths announced, pointer absent
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_NULL


def test_present_pairs_and_past_rules():
    B, Nkv, T, H = 2, 2, 8, 64
    pk = torch.zeros(B, Nkv, T, H, dtype=torch.bfloat16)
    assert code(base(present_k=pk)) == sdpa.SDPA_ERR_INVALID
    p, keep = base(P=4)
    p.past_k = sdpa.sdpa_view(None, 0, 0, 0)
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_SHAPE
    p, keep = base(past_k=torch.zeros(2, 2, 3, 64, dtype=torch.bfloat16),
                   past_v=torch.zeros(2, 2, 3, 64, dtype=torch.bfloat16))
    p.P = 0
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_SHAPE


def test_misaligned_pointer_and_stride():
    p, keep = base()
    p.q.data += 2                       # one bf16 element: not 16-byte aligned
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_ALIGNMENT
    p, keep = base()
    p.k.stride_s = 68                   # not a multiple of 8 elements
    p.k.stride_n = 68 * 8
    p.k.stride_b = 68 * 8 * 2
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_ALIGNMENT


def test_outputs_must_not_alias_inputs():
    B, Nq, S, H = 2, 4, 8, 64
    q = torch.zeros(B, Nq, S, H, dtype=torch.bfloat16)
    k = torch.zeros(B, 2, 8, H, dtype=torch.bfloat16)
    v = torch.zeros(B, 2, 8, H, dtype=torch.bfloat16)
    p, keep = sdpa.make_params(q, k, v, y=q)        # in place over q
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_ALIAS
    pres = torch.zeros(B, 2, 8, H, dtype=torch.bfloat16)
    p, keep = sdpa.make_params(q, k, v, y=torch.zeros_like(q), present_k=k, present_v=pres)
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_ALIAS   # shared past/present buffer
    p, keep = sdpa.make_params(q, k, v, y=torch.zeros_like(q), present_k=pres, present_v=pres)
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_ALIAS


def test_decode_limits():
    assert code(base(S=17, L=17), sdpa.SDPA_OP_DECODE) == sdpa.SDPA_ERR_UNSUPPORTED
    assert code(base(S=1, L=1, H=128, Hv=64), sdpa.SDPA_OP_DECODE) == sdpa.SDPA_ERR_UNSUPPORTED


def test_negative_sizes_and_overflow():
    p, keep = base()
    p.S = -1
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_SHAPE
    p, keep = base()
    p.q.stride_b = 1 << 50
    assert sdpa.sdpa_validate(p, 0) == sdpa.SDPA_ERR_OVERFLOW


def test_workspace_queries_are_host_only():
    p, keep = base(S=1, L=1, P=100, H=128, Hv=128, dtype=torch.float16)
    assert sdpa.sdpa_workspace_size(p, sdpa.SDPA_OP_DECODE) > 0
    bad, keep2 = base(window=0, causal="upper_left")
    assert sdpa.sdpa_workspace_size(bad, sdpa.SDPA_OP_FWD) == 0


def test_entry_points_reject_before_any_launch():
    bad, keep = base(window=0, causal="upper_left")
    assert sdpa.lib().sdpa_attn_fwd(ctypes.byref(bad), None, 0, None) == sdpa.SDPA_ERR_INVALID
    assert sdpa.lib().sdpa_attn_decode(ctypes.byref(bad), None, 0, None) == sdpa.SDPA_ERR_INVALID
    assert "window" in sdpa.sdpa_last_error()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_valid_call_without_a_gpu_fails_loudly():
    params, keep = base()
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa._check(sdpa.lib().sdpa_attn_fwd(ctypes.byref(params), None, 0, None))
    assert e.value.code == sdpa.SDPA_ERR_CUDA


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(sdpa, "_lib", None)
    monkeypatch.setattr(sdpa, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        sdpa.lib()


def test_kv_concat_rejections():
    cur = torch.zeros(2, 2, 3, 64, dtype=torch.float16)
    pres = torch.zeros(2, 2, 5, 64, dtype=torch.float16)
    L = sdpa.lib()
    keep = []
    v = lambda t: sdpa._view(t, keep)
    # P=2 but no past
    assert L.sdpa_kv_concat(1, 2, 2, 2, 3, 64, v(None), v(cur), None, v(pres), None) == sdpa.SDPA_ERR_SHAPE
    # present over the input
    assert L.sdpa_kv_concat(1, 2, 2, 0, 3, 64, v(None), v(cur), None, v(cur), None) == sdpa.SDPA_ERR_ALIAS
    # D not a multiple of 8
    assert L.sdpa_kv_concat(1, 2, 2, 0, 3, 12, v(None), v(cur), None, v(pres), None) == sdpa.SDPA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ rotary embedding

def _rot_args(dtype=1, B=2, N=2, S=4, D=64, R=0, inter=0, max_pos=16, ids=True, x=None, y=None):
    keep = []
    x = torch.zeros(B, N, S, D, dtype=torch.float16) if x is None else x
    y = torch.zeros(B, N, S, D, dtype=torch.float16) if y is None else y
    cos = torch.zeros(max(max_pos, 1), 32, dtype=torch.float16)
    pid = torch.zeros(B, S, dtype=torch.int64)
    keep += [x, y, cos, pid]
    return (dtype, B, N, S, D, sdpa._view(x, keep), sdpa._view(y, keep), cos.data_ptr(), cos.data_ptr(),
            max_pos, pid.data_ptr() if ids else None, R, inter, None), keep


def test_rotary_rejections():
    L = sdpa.lib()
    def rc(**kw):
        args, keep = _rot_args(**kw)
        return L.sdpa_rotary(*args)
    assert rc(dtype=7) == sdpa.SDPA_ERR_INVALID
    assert rc(R=7) == sdpa.SDPA_ERR_INVALID                 # odd
    assert rc(R=66) == sdpa.SDPA_ERR_INVALID                # wider than the head
    assert rc(inter=2) == sdpa.SDPA_ERR_INVALID
    assert rc(ids=False) == sdpa.SDPA_ERR_SHAPE             # rank-3 caches need max_pos == B*S
    assert rc(max_pos=0) == sdpa.SDPA_ERR_SHAPE
    x = torch.zeros(2, 2, 5, 64, dtype=torch.float16)
    assert rc(x=x[:, :, :4], y=x[:, :, 1:]) == sdpa.SDPA_ERR_ALIAS   # partial overlap
    args, keep = _rot_args()
    args = list(args)
    args[7] = None
    assert L.sdpa_rotary(*args) == sdpa.SDPA_ERR_NULL
    assert "NULL" in sdpa.sdpa_last_error()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_rotary_valid_call_without_a_gpu_fails_loudly():
    args, keep = _rot_args()
    assert sdpa.lib().sdpa_rotary(*args) == sdpa.SDPA_ERR_CUDA


def test_rotary_params_validation_and_workspace():
    cos = torch.zeros(64, 32, dtype=torch.bfloat16)
    assert code(base(rotary_cos=cos, rotary_sin=cos)) == sdpa.SDPA_OK
    p, keep = base(rotary_cos=cos, rotary_sin=cos)
    p.rotary_sin = None
    assert sdpa.sdpa_validate(p) == sdpa.SDPA_ERR_INVALID               # cos without sin
    assert code(base(rotary_cos=cos, rotary_sin=cos, rotary_dim=5)) == sdpa.SDPA_ERR_INVALID
    assert code(base(rotary_cos=cos, rotary_sin=cos, rotary_dim=66)) == sdpa.SDPA_ERR_INVALID
    qb = torch.zeros(4 * 64, dtype=torch.bfloat16)
    assert code(base(rotary_cos=cos, rotary_sin=cos, q_bias=qb)) == sdpa.SDPA_ERR_UNSUPPORTED
    plain, k1 = base(S=1, L=1, P=40, dtype=torch.float16)
    cos16 = torch.zeros(64, 32, dtype=torch.float16)
    rot, k2 = base(S=1, L=1, P=40, dtype=torch.float16, rotary_cos=cos16, rotary_sin=cos16)
    for op in (sdpa.SDPA_OP_FWD, sdpa.SDPA_OP_DECODE):
        assert sdpa.sdpa_workspace_size(rot, op) > sdpa.sdpa_workspace_size(plain, op)
    assert sdpa.lib().sdpa_attn_decode_static(ctypes.byref(rot), None) == sdpa.SDPA_ERR_UNSUPPORTED
    y = torch.zeros(2, 4, 8, 64, dtype=torch.bfloat16)
    p, keep = base(rotary_cos=cos, rotary_sin=cos)
    p.y = sdpa._view(y, keep)
    p.rotary_cos = p.rotary_sin = y.data_ptr()                           # output over the cache
    assert sdpa.sdpa_validate(p) == sdpa.SDPA_ERR_ALIAS


# ------------------------------------------------------------------ qk output

def test_qk_output_validation():
    qk = torch.zeros(2, 4, 8, 8, dtype=torch.float32)
    assert code(base(qk_out=qk, qk_mode=3)) == sdpa.SDPA_OK
    assert code(base(qk_out=qk, qk_mode=4)) == sdpa.SDPA_ERR_INVALID
    assert code(base(qk_out=qk, qk_mode=-1)) == sdpa.SDPA_ERR_INVALID
    assert code(base(qk_out=qk), sdpa.SDPA_OP_DECODE) == sdpa.SDPA_ERR_UNSUPPORTED
    # qk output over an input
    q = torch.zeros(2, 4, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, 8, 64, dtype=torch.bfloat16)
    v = torch.zeros(2, 2, 8, 64, dtype=torch.bfloat16)
    y = torch.zeros(2, 4, 8, 64, dtype=torch.bfloat16)
    over = q.view(torch.float32)[..., :8]                    # inside q's bytes
    p, keep = sdpa.make_params(q, k, v, y=y, qk_out=over)
    assert sdpa.sdpa_validate(p) == sdpa.SDPA_ERR_ALIAS


# ----------------------------------------------------------------- backward (host checks only)

def test_backward_subset_validates():
    assert code(base(), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(H=128, Hv=128, causal="lower_right", window=4), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(causal="upper_left", lens=torch.tensor([3, 8]), len_kind="nonpad"), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(dtype=torch.float16, head_sink=torch.zeros(4, dtype=torch.float16)), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK


@pytest.mark.parametrize("kw,why", [
    (dict(softcap=30.0), "softcap"),
    (dict(dtype=torch.float32, H=64, Hv=64), "f32"),
    (dict(H=96, Hv=96), "head size"),
    (dict(H=64, Hv=128), "H != Hv"),
])
def test_backward_rejects_outside_its_subset(kw, why):
    assert code(base(**kw), sdpa.SDPA_OP_BWD) == sdpa.SDPA_ERR_UNSUPPORTED, why


def test_backward_takes_masks_and_key_lengths():
    assert code(base(keep_mask=torch.ones(1, 1, 8, 8, dtype=torch.uint8), keep_kind="bool"), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(add_mask=torch.zeros(1, 1, 8, 8, dtype=torch.bfloat16)), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(lens=torch.tensor([3, 8], dtype=torch.int32), len_kind="keylen"), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK


def test_backward_takes_past_rows_and_projection_biases():
    assert code(base(P=5), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK
    assert code(base(q_bias=torch.zeros(4 * 64, dtype=torch.bfloat16), k_bias=torch.zeros(2 * 64, dtype=torch.bfloat16),
                     v_bias=torch.zeros(2 * 64, dtype=torch.bfloat16)), sdpa.SDPA_OP_BWD) == sdpa.SDPA_OK


def test_backward_rejects_present_outputs():
    pk = torch.zeros(2, 2, 8, 64, dtype=torch.bfloat16)
    pv = torch.zeros(2, 2, 8, 64, dtype=torch.bfloat16)
    assert code(base(present_k=pk, present_v=pv), sdpa.SDPA_OP_BWD) == sdpa.SDPA_ERR_INVALID


def test_backward_workspace_is_two_floats_per_query_row():
    params, _keep = base(B=3, Nq=4, S=100)
    assert sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_BWD) == 2 * ((3 * 4 * 100 * 4 + 255) // 256 * 256)
    params, _keep = base(softcap=5.0)
    assert sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_BWD) == 0


def test_backward_workspace_holds_the_materialised_rows():
    """Past rows or k / v biases add contiguous copies of the T key and value rows; a q bias
    adds a copy of the biased query."""
    a = lambda n: (n + 255) // 256 * 256
    stats = 2 * a(2 * 4 * 8 * 4)
    params, _keep = base(P=5)
    assert sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_BWD) == stats + 2 * a(2 * 2 * 13 * 64 * 2)
    params, _keep = base(q_bias=torch.zeros(4 * 64, dtype=torch.bfloat16))
    assert sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_BWD) == stats + a(2 * 4 * 8 * 64 * 2)


def test_backward_gradient_alias_is_rejected_before_launch():
    """dq overlapping q is refused on the host (no device work is enqueued)."""
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    v = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    dy = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_attn_bwd(q, k, v, dy, dq=q, workspace=torch.zeros(4096, dtype=torch.uint8), stream=0)
    assert e.value.code == sdpa.SDPA_ERR_ALIAS
