"""Python binding of libsdpa.so (argument marshalling only).

The functions here carry the names of the C entry points declared in include/sdpa.h and
do nothing but turn torch tensors into the C structs, pick the caller's current CUDA
stream, and raise on a non-zero status.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback of any kind: if libsdpa.so is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdpa.so")

# status codes (include/sdpa.h)
SDPA_OK = 0
SDPA_ERR_INVALID = 1
SDPA_ERR_BOUNDS = 11
SDPA_ERR_SHAPE = 2
SDPA_ERR_UNSUPPORTED = 3
SDPA_ERR_ALIGNMENT = 4
SDPA_ERR_ALIAS = 5
SDPA_ERR_OVERFLOW = 6
SDPA_ERR_WORKSPACE = 7
SDPA_ERR_CUDA = 8
SDPA_ERR_TIMEOUT = 9
SDPA_ERR_NULL = 10

SDPA_F32, SDPA_F16, SDPA_BF16 = 0, 1, 2
SDPA_CAUSAL_NONE, SDPA_CAUSAL_UPPER_LEFT, SDPA_CAUSAL_LOWER_RIGHT = 0, 1, 2
SDPA_KEEP_NONE, SDPA_KEEP_BOOL_U8, SDPA_KEEP_FILTER_I32 = 0, 1, 2
SDPA_LEN_NONE, SDPA_LEN_NONPAD_I64, SDPA_LEN_KEYLEN_I32, SDPA_LEN_SEQLENS_K_I32 = 0, 1, 2, 3
SDPA_OP_FWD, SDPA_OP_DECODE, SDPA_OP_BWD = 0, 1, 2

_DTYPES = {torch.float32: SDPA_F32, torch.float16: SDPA_F16, torch.bfloat16: SDPA_BF16}
CAUSAL = {"none": SDPA_CAUSAL_NONE, "upper_left": SDPA_CAUSAL_UPPER_LEFT,
          "lower_right": SDPA_CAUSAL_LOWER_RIGHT}
KEEP = {"none": SDPA_KEEP_NONE, "bool": SDPA_KEEP_BOOL_U8, "filter": SDPA_KEEP_FILTER_I32}
LENS = {"none": SDPA_LEN_NONE, "nonpad": SDPA_LEN_NONPAD_I64, "keylen": SDPA_LEN_KEYLEN_I32,
        "seqlens_k": SDPA_LEN_SEQLENS_K_I32}


class SdpaError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"sdpa error {code}: {message}")
        self.code = code


class sdpa_view(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_n", ctypes.c_int64), ("stride_s", ctypes.c_int64)]


class sdpa_params(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_int32),
        ("B", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Nkv", ctypes.c_int32),
        ("S", ctypes.c_int32), ("L", ctypes.c_int32), ("P", ctypes.c_int32),
        ("H", ctypes.c_int32), ("Hv", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("q", sdpa_view), ("k", sdpa_view), ("v", sdpa_view),
        ("past_k", sdpa_view), ("past_v", sdpa_view),
        ("present_k", sdpa_view), ("present_v", sdpa_view), ("y", sdpa_view),
        ("q_bias", ctypes.c_void_p), ("k_bias", ctypes.c_void_p), ("v_bias", ctypes.c_void_p),
        ("head_sink", ctypes.c_void_p),
        ("has_scale", ctypes.c_int32), ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("causal", ctypes.c_int32), ("window", ctypes.c_int64),
        ("add_mask", sdpa_view), ("add_mask_dtype", ctypes.c_int32), ("add_mask_T", ctypes.c_int64),
        ("keep_mask", sdpa_view), ("keep_kind", ctypes.c_int32), ("keep_mask_T", ctypes.c_int64),
        ("len_kind", ctypes.c_int32), ("lens", ctypes.c_void_p),
        ("mask_filter_value", ctypes.c_float),
        ("softcap_before_bias", ctypes.c_int32),
        ("rotary_cos", ctypes.c_void_p), ("rotary_sin", ctypes.c_void_p),
        ("rotary_max_pos", ctypes.c_int64), ("rotary_dim", ctypes.c_int32),
        ("rotary_interleaved", ctypes.c_int32),
        ("qk_out", sdpa_view), ("qk_mode", ctypes.c_int32),
    ]


EXPORTED = ("sdpa_attn_fwd", "sdpa_attn_decode", "sdpa_workspace_size", "sdpa_validate",
            "sdpa_kv_concat", "sdpa_query_status", "sdpa_last_error", "sdpa_last_kernel_name",
            "sdpa_version", "sdpa_launch_count", "sdpa_attn_decode_static", "sdpa_rotary",
            "sdpa_attn_bwd")

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libsdpa.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(sdpa_params)
        L.sdpa_attn_fwd.argtypes = [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.sdpa_attn_fwd.restype = ctypes.c_int
        L.sdpa_attn_decode.argtypes = [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.sdpa_attn_decode.restype = ctypes.c_int
        L.sdpa_attn_bwd.argtypes = [P, sdpa_view, sdpa_view, sdpa_view, sdpa_view, ctypes.c_void_p,
                                    ctypes.c_size_t, ctypes.c_void_p]
        L.sdpa_attn_bwd.restype = ctypes.c_int
        L.sdpa_attn_decode_static.argtypes = [P, ctypes.c_void_p]
        L.sdpa_attn_decode_static.restype = ctypes.c_int
        L.sdpa_workspace_size.argtypes = [P, ctypes.c_int]
        L.sdpa_workspace_size.restype = ctypes.c_size_t
        L.sdpa_validate.argtypes = [P, ctypes.c_int]
        L.sdpa_validate.restype = ctypes.c_int
        L.sdpa_kv_concat.argtypes = [ctypes.c_int] + [ctypes.c_int32] * 5 + \
            [sdpa_view, sdpa_view, ctypes.c_void_p, sdpa_view, ctypes.c_void_p]
        L.sdpa_kv_concat.restype = ctypes.c_int
        L.sdpa_rotary.argtypes = [ctypes.c_int] + [ctypes.c_int32] * 4 + \
            [sdpa_view, sdpa_view, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
             ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        L.sdpa_rotary.restype = ctypes.c_int
        L.sdpa_query_status.argtypes = [ctypes.c_void_p]
        L.sdpa_query_status.restype = ctypes.c_int
        for f in ("sdpa_last_error", "sdpa_last_kernel_name", "sdpa_version"):
            getattr(L, f).restype = ctypes.c_char_p
            getattr(L, f).argtypes = []
        L.sdpa_launch_count.restype = ctypes.c_int64
        L.sdpa_launch_count.argtypes = []
        _lib = L
    return _lib


def sdpa_last_error() -> str:
    return lib().sdpa_last_error().decode()


def sdpa_last_kernel_name() -> str:
    return lib().sdpa_last_kernel_name().decode()


def sdpa_version() -> str:
    return lib().sdpa_version().decode()


def sdpa_launch_count() -> int:
    return int(lib().sdpa_launch_count())


def _check(rc: int):
    if rc != SDPA_OK:
        raise SdpaError(rc, sdpa_last_error())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _view(t: Optional[torch.Tensor], keep: list) -> sdpa_view:
    if t is None:
        return sdpa_view(None, 0, 0, 0)
    if t.dim() != 4:
        raise ValueError("views are 4-D (batch, heads, seq, dim)")
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError("the last dimension must be contiguous")
    keep.append(t)
    sb, sh, ss, _ = t.stride()
    return sdpa_view(t.data_ptr(), sb, sh, ss)


def _ptr(t: Optional[torch.Tensor], keep: list):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("1-D parameter tensors must be contiguous")
    keep.append(t)
    return t.data_ptr()


def _mask4(m: Optional[torch.Tensor], B: int, Nq: int, S: int) -> Optional[torch.Tensor]:
    """Broadcast a mask of rank 2..4 (right-aligned, ONNX style) to a (B, Nq, S, Tm) view."""
    if m is None:
        return None
    while m.dim() < 4:
        m = m.unsqueeze(0)
    return m.expand(B, Nq, S, m.shape[-1])


def make_params(q, k, v, *, y=None, past_k=None, past_v=None, present_k=None, present_v=None,
                q_bias=None, k_bias=None, v_bias=None, head_sink=None, scale=None, softcap=0.0,
                causal="none", window=-1, add_mask=None, keep_mask=None, keep_kind="none",
                lens=None, len_kind="none", mask_filter_value=-10000.0,
                softcap_before_bias=False, rotary_cos=None, rotary_sin=None, rotary_dim=0,
                rotary_interleaved=False, qk_out=None, qk_mode=0) -> Tuple[sdpa_params, list]:
    """Fills sdpa_params from 4-D (B, N, S, D) views.  Returns (params, tensors to keep alive)."""
    keep: list = []
    p = sdpa_params()
    p.struct_size = ctypes.sizeof(sdpa_params)
    B, Nq, S, H = q.shape
    Nkv, L, Hv = k.shape[1], k.shape[2], v.shape[3]
    P = 0 if past_k is None else past_k.shape[2]
    p.B, p.Nq, p.Nkv, p.S, p.L, p.P, p.H, p.Hv = B, Nq, Nkv, S, L, P, H, Hv
    p.dtype = _DTYPES[q.dtype]
    p.q, p.k, p.v = _view(q, keep), _view(k, keep), _view(v, keep)
    p.past_k, p.past_v = _view(past_k, keep), _view(past_v, keep)
    p.present_k, p.present_v = _view(present_k, keep), _view(present_v, keep)
    p.y = _view(y, keep)
    p.q_bias, p.k_bias, p.v_bias = _ptr(q_bias, keep), _ptr(k_bias, keep), _ptr(v_bias, keep)
    p.head_sink = _ptr(head_sink, keep)
    p.has_scale = 0 if scale is None else 1
    p.scale = 0.0 if scale is None else float(scale)
    p.softcap = float(softcap)
    p.causal = CAUSAL[causal] if isinstance(causal, str) else int(causal)
    p.window = int(window)
    am = _mask4(add_mask, B, Nq, S)
    p.add_mask = _view(am, keep)
    p.add_mask_dtype = _DTYPES[am.dtype] if am is not None else 0
    p.add_mask_T = 0 if am is None else am.shape[-1]
    km = _mask4(keep_mask, B, Nq, S)
    p.keep_mask = _view(km, keep)
    p.keep_kind = (KEEP[keep_kind] if isinstance(keep_kind, str) else int(keep_kind)) if km is not None else 0
    p.keep_mask_T = 0 if km is None else km.shape[-1]
    p.len_kind = (LENS[len_kind] if isinstance(len_kind, str) else int(len_kind)) if lens is not None else 0
    p.lens = _ptr(lens, keep)
    p.mask_filter_value = float(mask_filter_value)
    p.softcap_before_bias = 1 if softcap_before_bias else 0
    if rotary_cos is not None:
        p.rotary_cos, p.rotary_sin = _ptr(rotary_cos, keep), _ptr(rotary_sin, keep)
        p.rotary_max_pos = rotary_cos.shape[0]
    p.rotary_dim = int(rotary_dim)
    p.rotary_interleaved = 1 if rotary_interleaved else 0
    p.qk_out = _view(qk_out, keep)
    p.qk_mode = int(qk_mode)
    return p, keep


def sdpa_validate(params: sdpa_params, op: int = SDPA_OP_FWD) -> int:
    return lib().sdpa_validate(ctypes.byref(params), op)


def sdpa_workspace_size(params: sdpa_params, op: int = SDPA_OP_FWD) -> int:
    return int(lib().sdpa_workspace_size(ctypes.byref(params), op))


def _workspace(params, op, workspace, device):
    need = sdpa_workspace_size(params, op)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def _run(entry, op, q, k, v, y, workspace, stream, kw):
    if y is None:
        y = torch.empty(q.shape[0], q.shape[1], q.shape[2], v.shape[3], dtype=q.dtype, device=q.device)
    params, keep = make_params(q, k, v, y=y, **kw)
    ws, nbytes = _workspace(params, op, workspace, q.device)
    _check(entry(ctypes.byref(params), None if ws is None else ws.data_ptr(), nbytes, _stream(stream)))
    return y


def sdpa_attn_fwd(q, k, v, *, y=None, workspace=None, stream=None, **kw) -> torch.Tensor:
    """Forward over 4-D (B, N, S, D) CUDA views; returns y (B, Nq, S, Hv) (a view if `y` is given).

    Keyword arguments are those of make_params (past/present, biases, head_sink, scale,
    softcap, causal, window, masks, lengths, mask_filter_value, softcap_before_bias)."""
    return _run(lib().sdpa_attn_fwd, SDPA_OP_FWD, q, k, v, y, workspace, stream, kw)


def mha_bias_segments(projection_bias: Optional[torch.Tensor], num_heads: int, H: int, Hv: int,
                      kv_rank: int):
    """(q_bias, k_bias, v_bias) for the C ABI from MultiHeadAttention's single projection-bias
    input ("Custom operators", Microsoft MultiHeadAttention): [query N*H | key N*H | value N*Hv];
    rank-4 key/value take no key/value segment (only the query segment applies).  Slices of
    the input: pointer offsets, no arithmetic."""
    if projection_bias is None:
        return None, None, None
    nq, nv = num_heads * H, num_heads * Hv
    if projection_bias.dim() != 1 or projection_bias.numel() != 2 * nq + nv:
        raise ValueError(f"projection bias of {2 * nq + nv} values expected, got {tuple(projection_bias.shape)}")
    segments = (projection_bias[:nq], projection_bias[nq:2 * nq], projection_bias[2 * nq:])
    if kv_rank == 4:
        return segments[0], None, None
    if kv_rank != 3:
        raise ValueError("key/value must be rank 3 or rank 4")
    return segments


def _heads4(t: torch.Tensor, num_heads: int) -> torch.Tensor:
    """(B, N, S, D) view of a rank-3 (B, S, N*D) tensor; rank-4 tensors pass through."""
    if t.dim() == 4:
        return t
    B, S, ND = t.shape
    return t.view(B, S, num_heads, ND // num_heads).permute(0, 2, 1, 3)


def sdpa_mha_fwd(query, key, value, *, num_heads: int, projection_bias=None, y=None, workspace=None,
                 stream=None, **kw) -> torch.Tensor:
    """MultiHeadAttention forward over the operator's tensors: query (B, S, N*H); key and value
    rank-3 (B, L, N*H) / (B, L, N*Hv) or rank-4 (B, N, L, H) / (B, N, L, Hv); projection_bias
    the operator's single (2*N*H + N*Hv,) input, of which rank-4 key/value take only the query
    segment.  Returns y (B, S, N*Hv).  Other keywords as sdpa_attn_fwd (masks, lengths,
    past/present, scale, causal / unidirectional, mask_filter_value)."""
    if key.dim() != value.dim() or key.dim() not in (3, 4):
        raise ValueError("key and value must both be rank 3 or both rank 4")
    q4, k4, v4 = _heads4(query, num_heads), _heads4(key, num_heads), _heads4(value, num_heads)
    B, N, S, H = q4.shape
    Hv = v4.shape[3]
    q_bias, k_bias, v_bias = mha_bias_segments(projection_bias, num_heads, H, Hv, key.dim())
    if y is None:
        y = torch.empty(B, S, N * Hv, dtype=query.dtype, device=query.device)
    sdpa_attn_fwd(q4, k4, v4, y=_heads4(y, num_heads), workspace=workspace, stream=stream,
                  q_bias=q_bias, k_bias=k_bias, v_bias=v_bias, **kw)
    return y


def sdpa_attn_decode(q, k, v, *, y=None, workspace=None, stream=None, **kw) -> torch.Tensor:
    """Split-KV decode (S <= 16), same arguments as sdpa_attn_fwd."""
    return _run(lib().sdpa_attn_decode, SDPA_OP_DECODE, q, k, v, y, workspace, stream, kw)


def sdpa_attn_decode_static(q, k, v, *, y=None, stream=None, **kw) -> torch.Tensor:
    """Decode without a workspace (the library's built-in device scratch), for callers
    that cannot allocate device memory; same arguments as sdpa_attn_decode otherwise, except
    that the caller passes the output y (B, Nq, S, Hv): like the C call, this binding
    allocates nothing.  Calls that overlap on the GPU share that scratch and race: keep them
    on one stream."""
    if y is None:
        raise ValueError("sdpa_attn_decode_static allocates nothing: pass the output y")
    params, keep = make_params(q, k, v, y=y, **kw)
    _check(lib().sdpa_attn_decode_static(ctypes.byref(params), _stream(stream)))
    return y


def sdpa_attn_bwd(q, k, v, dy, *, dq=None, dk=None, dv=None, workspace=None, stream=None, **kw):
    """Backward over 4-D (B, N, S, D) CUDA views: returns (dq, dk, dv) for the upstream
    gradient dy (B, Nq, S, Hv).  Keyword arguments describe the forward problem as for
    sdpa_attn_fwd (past_k / past_v, projection biases, masks, lengths, head_sink, scale,
    causal, window).  dk and dv cover the P past rows followed by the L new rows."""
    B, Nq, S, H = q.shape
    Nkv, L, Hv = k.shape[1], k.shape[2], v.shape[3]
    past_k = kw.get("past_k")
    T = L + (0 if past_k is None else past_k.shape[2])
    if dq is None:
        dq = torch.empty(B, Nq, S, H, dtype=q.dtype, device=q.device)
    if dk is None:
        dk = torch.empty(B, Nkv, T, H, dtype=q.dtype, device=q.device)
    if dv is None:
        dv = torch.empty(B, Nkv, T, Hv, dtype=q.dtype, device=q.device)
    params, keep = make_params(q, k, v, **kw)
    ws, nbytes = _workspace(params, SDPA_OP_BWD, workspace, q.device)
    _check(lib().sdpa_attn_bwd(ctypes.byref(params), _view(dy, keep), _view(dq, keep), _view(dk, keep),
                               _view(dv, keep), None if ws is None else ws.data_ptr(), nbytes, _stream(stream)))
    return dq, dk, dv


def sdpa_kv_concat(past: Optional[torch.Tensor], cur: torch.Tensor, present: torch.Tensor,
                   bias: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """present[:, :, :P] = past; present[:, :, P:] = cur (+ bias), all (B, N, S, D) views."""
    keep: list = []
    B, N, L, D = cur.shape
    P = 0 if past is None else past.shape[2]
    rc = lib().sdpa_kv_concat(_DTYPES[cur.dtype], B, N, P, L, D, _view(past, keep), _view(cur, keep),
                              _ptr(bias, keep), _view(present, keep), _stream(stream))
    _check(rc)
    return present


def sdpa_rotary(x: torch.Tensor, cos_cache: torch.Tensor, sin_cache: torch.Tensor,
                position_ids: Optional[torch.Tensor] = None, *, rotary_dim: int = 0,
                interleaved: bool = False, num_heads: Optional[int] = None,
                y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """RotaryEmbedding over a rank-4 (B, N, S, D) or rank-3 (B, S, N*D) tensor (num_heads
    given).  cos/sin caches: rank-2 (max_pos, R/2) with position_ids (B, S) int64, or rank-3
    (B, S, R/2) without.  Returns y in x's shape (`y` may be x itself)."""
    keep: list = []
    if x.dim() == 3:
        if not num_heads:
            raise ValueError("a rank-3 input needs num_heads")
        B, S, hidden = x.shape
        x4 = x.view(B, S, num_heads, hidden // num_heads).transpose(1, 2)
    else:
        x4 = x
    B, N, S, D = x4.shape
    if y is None:
        y = torch.empty_like(x)
    y4 = y.view(B, S, N, D).transpose(1, 2) if y.dim() == 3 else y
    if cos_cache.dim() == 3:
        max_pos = cos_cache.shape[0] * cos_cache.shape[1]
    else:
        max_pos = cos_cache.shape[0]
    pos = None
    if position_ids is not None:
        pos = position_ids.to(torch.int64).expand(B, S).contiguous()
    rc = lib().sdpa_rotary(_DTYPES[x.dtype], B, N, S, D, _view(x4, keep), _view(y4, keep),
                           _ptr(cos_cache, keep), _ptr(sin_cache, keep), max_pos, _ptr(pos, keep),
                           int(rotary_dim), 1 if interleaved else 0, _stream(stream))
    _check(rc)
    return y


def sdpa_query_status(stream=None) -> int:
    return int(lib().sdpa_query_status(_stream(stream)))


# ----------------------------------------------------------------------------------------
# Workload cases (scaled_dot_product_gb300.workloads.Case) through the entry points
# ----------------------------------------------------------------------------------------

def case_kwargs(case, present_k=None, present_v=None) -> dict:
    """make_params keyword arguments for a workload case already on the device."""
    return dict(past_k=case.past_k, past_v=case.past_v, present_k=present_k, present_v=present_v,
                q_bias=case.q_bias, k_bias=case.k_bias, v_bias=case.v_bias,
                head_sink=case.head_sink, scale=case.scale, softcap=case.softcap,
                causal=case.causal, window=case.window, add_mask=case.add_mask,
                keep_mask=case.keep_mask, keep_kind=case.keep_kind, lens=case.lens,
                len_kind=case.len_kind, mask_filter_value=case.mask_filter_value,
                softcap_before_bias=case.softcap_before_bias, rotary_cos=case.rotary_cos,
                rotary_sin=case.rotary_sin, rotary_dim=case.rotary_dim,
                rotary_interleaved=case.rotary_interleaved)


def case_outputs(case):
    """Allocates y in the layout of the query (rank-3 or rank-4) and present if wanted."""
    dev = case.q.device
    y_store = torch.empty(case.y_shape(), dtype=case.dtype, device=dev)
    from .workloads import as4d
    y4 = as4d(y_store, case.q_layout, case.Nq)
    pk = pv = None
    if case.want_present:
        pk = torch.empty(case.B, case.Nkv, case.T, case.H, dtype=case.dtype, device=dev)
        pv = torch.empty(case.B, case.Nkv, case.T, case.Hv, dtype=case.dtype, device=dev)
    return y_store, y4, pk, pv


def run_case(case, op: str = "fwd", outputs=None, workspace=None, stream=None, **extra):
    """Runs a device-resident case; returns (y in the query's layout, present_k, present_v).
    `extra` adds make_params keywords (e.g. qk_out / qk_mode)."""
    q, k, v = case.views()
    y_store, y4, pk, pv = outputs if outputs is not None else case_outputs(case)
    entry = sdpa_attn_decode if op == "decode" else sdpa_attn_fwd
    entry(q, k, v, y=y4, workspace=workspace, stream=stream, **case_kwargs(case, pk, pv), **extra)
    return y_store, pk, pv


def case_workspace(case, op: str = "fwd") -> Optional[torch.Tensor]:
    """Device workspace for running `case` through `op`, or None when none is needed."""
    need = _workspace_need(case, op)
    return None if need == 0 else torch.empty(need, dtype=torch.uint8, device=case.q.device)


def _workspace_need(case, op: str) -> int:
    q, k, v = case.views()
    y_store, y4, pk, pv = case_outputs(case)
    params, keep = make_params(q, k, v, y=y4, **case_kwargs(case, pk, pv))
    return sdpa_workspace_size(params, SDPA_OP_DECODE if op == "decode" else SDPA_OP_FWD)
