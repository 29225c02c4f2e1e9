"""Double-precision CPU oracle for scaled dot-product attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module only
marshals torch CPU tensors (any 4-D strided view with a contiguous last dimension) into
its parameter struct.  What it computes follows the onnx-light documentation pages:
``include_nn_kernels.h`` (class Attention), and the "Custom operators" page sections
Microsoft MultiHeadAttention and Microsoft GroupQueryAttention.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

F32, F16, BF16, U8, I32, I64, F64 = 0, 1, 2, 3, 4, 5, 6
CAUSAL_NONE, CAUSAL_UPPER_LEFT, CAUSAL_LOWER_RIGHT = 0, 1, 2
KEEP_NONE, KEEP_BOOL, KEEP_FILTER = 0, 1, 2
LEN_NONE, LEN_NONPAD_I64, LEN_KEYLEN_I32, LEN_SEQLENS_K_I32 = 0, 1, 2, 3

_DT = {
    torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.uint8: U8,
    torch.bool: U8, torch.int32: I32, torch.int64: I64, torch.float64: F64,
}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no SIMD flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("sb", ctypes.c_int64), ("sh", ctypes.c_int64), ("ss", ctypes.c_int64)]


class _Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Nq", ctypes.c_int32), ("Nkv", ctypes.c_int32), ("S", ctypes.c_int32),
        ("L", ctypes.c_int32), ("P", ctypes.c_int32), ("H", ctypes.c_int32), ("Hv", ctypes.c_int32),
        ("q", _Tensor), ("k", _Tensor), ("v", _Tensor), ("past_k", _Tensor), ("past_v", _Tensor),
        ("q_bias", ctypes.c_void_p), ("k_bias", ctypes.c_void_p), ("v_bias", ctypes.c_void_p),
        ("bias_dtype", ctypes.c_int32),
        ("scale", ctypes.c_double), ("softcap", ctypes.c_double),
        ("causal", ctypes.c_int32), ("window", ctypes.c_int64),
        ("head_sink", ctypes.c_void_p),
        ("add_mask", _Tensor), ("add_mask_T", ctypes.c_int64),
        ("keep_mask", _Tensor), ("keep_kind", ctypes.c_int32), ("keep_mask_T", ctypes.c_int64),
        ("len_kind", ctypes.c_int32), ("lens", ctypes.c_void_p),
        ("mask_filter_value", ctypes.c_double),
        ("softcap_before_bias", ctypes.c_int32),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB_OVERRIDE lets the mutation test load a deliberately broken build
        override = os.environ.get("ORACLE_LIB_OVERRIDE")
        _lib = ctypes.CDLL(override if override else build())
        _lib.oracle_attention_rows.restype = ctypes.c_int
        _lib.oracle_attention_rows.argtypes = [ctypes.POINTER(_Params), ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        _lib.oracle_qk_rows.restype = ctypes.c_int
        _lib.oracle_qk_rows.argtypes = [ctypes.POINTER(_Params), ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        _lib.oracle_attention_backward.restype = ctypes.c_int
        _lib.oracle_attention_backward.argtypes = [ctypes.POINTER(_Params), ctypes.POINTER(_Tensor), ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _lib.oracle_present.restype = ctypes.c_int
        _lib.oracle_present.argtypes = [ctypes.c_int32] * 6 + [ctypes.POINTER(_Tensor)] * 2 + \
            [ctypes.c_void_p, ctypes.c_void_p]
        _lib.oracle_rotary.restype = ctypes.c_int
        _lib.oracle_rotary.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(_Tensor), ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        _lib.oracle_to_double.restype = ctypes.c_double
        _lib.oracle_to_double.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64]
        _lib.oracle_round_f16.restype = ctypes.c_uint16
        _lib.oracle_round_f16.argtypes = [ctypes.c_double]
        _lib.oracle_round_bf16.restype = ctypes.c_uint16
        _lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        _lib.oracle_round_array.restype = ctypes.c_int
        _lib.oracle_round_array.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    return _lib


def _view(t: Optional[torch.Tensor], keep: list) -> _Tensor:
    """A 4-D CPU tensor (b, h, s, d) with stride(-1) == 1 (other strides may be 0)."""
    if t is None:
        return _Tensor(None, 0, 0, 0, 0)
    assert t.device.type == "cpu" and t.dim() == 4 and (t.shape[-1] <= 1 or t.stride(-1) == 1), \
        "oracle tensors: 4-D CPU views with a contiguous last dimension"
    keep.append(t)
    sb, sh, ss, _ = t.stride()
    return _Tensor(t.data_ptr(), _DT[t.dtype], sb, sh, ss)


def _ptr(t: Optional[torch.Tensor], keep: list):
    if t is None:
        return None
    t = t.contiguous()
    keep.append(t)
    return t.data_ptr()


@dataclass
class Problem:
    """One attention problem in oracle terms.  Every tensor is a torch CPU tensor.

    q (B,Nq,S,H); k (B,Nkv,L,H); v (B,Nkv,L,Hv); past_k/past_v (B,Nkv,P,H/Hv) or None;
    add_mask / keep_mask: 4-D views broadcastable by stride to (B,Nq,S,Tm);
    lens: (B,) int64 for nonpad, int32 for key lengths and seqlens_k.
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    past_k: Optional[torch.Tensor] = None
    past_v: Optional[torch.Tensor] = None
    q_bias: Optional[torch.Tensor] = None
    k_bias: Optional[torch.Tensor] = None
    v_bias: Optional[torch.Tensor] = None
    scale: Optional[float] = None
    softcap: float = 0.0
    causal: int = CAUSAL_NONE
    window: int = -1
    head_sink: Optional[torch.Tensor] = None
    add_mask: Optional[torch.Tensor] = None
    keep_mask: Optional[torch.Tensor] = None
    keep_kind: int = KEEP_NONE
    len_kind: int = LEN_NONE
    lens: Optional[torch.Tensor] = None
    mask_filter_value: float = -10000.0
    softcap_before_bias: bool = False

    @property
    def dims(self):
        B, Nq, S, H = self.q.shape
        Nkv, L, Hv = self.k.shape[1], self.k.shape[2], self.v.shape[3]
        P = 0 if self.past_k is None else self.past_k.shape[2]
        return B, Nq, Nkv, S, L, P, H, Hv


def _params(pr: Problem, keep: list) -> _Params:
    B, Nq, Nkv, S, L, P, H, Hv = pr.dims
    p = _Params()
    p.B, p.Nq, p.Nkv, p.S, p.L, p.P, p.H, p.Hv = B, Nq, Nkv, S, L, P, H, Hv
    p.q, p.k, p.v = _view(pr.q, keep), _view(pr.k, keep), _view(pr.v, keep)
    p.past_k, p.past_v = _view(pr.past_k, keep), _view(pr.past_v, keep)
    p.q_bias, p.k_bias, p.v_bias = _ptr(pr.q_bias, keep), _ptr(pr.k_bias, keep), _ptr(pr.v_bias, keep)
    bias_src = next((t for t in (pr.q_bias, pr.k_bias, pr.v_bias, pr.head_sink) if t is not None), None)
    p.bias_dtype = _DT[bias_src.dtype] if bias_src is not None else _DT[pr.q.dtype]
    p.scale = (1.0 / math.sqrt(H)) if pr.scale is None else float(pr.scale)
    p.softcap = float(pr.softcap)
    p.causal = int(pr.causal)
    p.window = int(pr.window)
    p.head_sink = _ptr(pr.head_sink, keep)
    p.add_mask = _view(pr.add_mask, keep)
    p.add_mask_T = 0 if pr.add_mask is None else pr.add_mask.shape[-1]
    p.keep_mask = _view(pr.keep_mask, keep)
    p.keep_kind = int(pr.keep_kind) if pr.keep_mask is not None else KEEP_NONE
    p.keep_mask_T = 0 if pr.keep_mask is None else pr.keep_mask.shape[-1]
    p.len_kind = int(pr.len_kind) if pr.lens is not None else LEN_NONE
    p.lens = _ptr(pr.lens, keep)
    p.mask_filter_value = float(pr.mask_filter_value)
    p.softcap_before_bias = int(bool(pr.softcap_before_bias))
    return p


def attention_rows(pr: Problem, rows: Sequence[Sequence[int]], nthreads: int = 0):
    """Output rows y[b, h, i, :] (float64, shape (len(rows), Hv)) and the thread count used."""
    keep: list = []
    p = _params(pr, keep)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((r.shape[0], p.Hv), dtype=np.float64)
    n = lib().oracle_attention_rows(ctypes.byref(p), r.ctypes.data, r.shape[0], out.ctypes.data,
                                    int(nthreads))
    if n < 0:
        raise ValueError(f"oracle rejected the problem (code {n})")
    return out, n


def qk_rows(pr: Problem, mode: int, rows: Sequence[Sequence[int]], nthreads: int = 0):
    """qk output rows (class Attention, qk_matmul_output_mode = mode) of the selected query
    rows: float64 (len(rows), T), and the thread count used."""
    keep: list = []
    p = _params(pr, keep)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    T = p.P + p.L
    out = np.zeros((r.shape[0], T), dtype=np.float64)
    n = lib().oracle_qk_rows(ctypes.byref(p), int(mode), r.ctypes.data, r.shape[0], out.ctypes.data,
                             int(nthreads))
    if n < 0:
        raise ValueError(f"oracle rejected the problem (code {n})")
    return out, n


def qk(pr: Problem, mode: int, nthreads: int = 0) -> np.ndarray:
    """Full qk output (B, Nq, S, T) in float64."""
    B, Nq, _, S, L, P, _, _ = pr.dims
    rows = np.stack(np.meshgrid(np.arange(B), np.arange(Nq), np.arange(S), indexing="ij"), -1)
    out, _ = qk_rows(pr, mode, rows.reshape(-1, 3), nthreads)
    return out.reshape(B, Nq, S, P + L)


def backward(pr: Problem, dy: torch.Tensor, nthreads: int = 0):
    """Gradients (dq, dk, dv) in float64 of the attention for the upstream gradient dy
    (B, Nq, S, Hv): shapes (B, Nq, S, H), (B, Nkv, P+L, H), (B, Nkv, P+L, Hv)."""
    keep: list = []
    p = _params(pr, keep)
    dyv = _view(dy, keep)
    T = p.P + p.L
    dq = np.zeros((p.B, p.Nq, p.S, p.H))
    dk = np.zeros((p.B, p.Nkv, T, p.H))
    dv = np.zeros((p.B, p.Nkv, T, p.Hv))
    n = lib().oracle_attention_backward(ctypes.byref(p), ctypes.byref(dyv), dq.ctypes.data, dk.ctypes.data,
                                        dv.ctypes.data, int(nthreads))
    if n < 0:
        raise ValueError(f"oracle rejected the problem (code {n})")
    return dq, dk, dv


def attention(pr: Problem, nthreads: int = 0) -> np.ndarray:
    """Full output (B, Nq, S, Hv) in float64."""
    B, Nq, _, S, _, _, _, Hv = pr.dims
    rows = np.stack(np.meshgrid(np.arange(B), np.arange(Nq), np.arange(S), indexing="ij"), -1)
    out, _ = attention_rows(pr, rows.reshape(-1, 3), nthreads)
    return out.reshape(B, Nq, S, Hv)


def mha_projection_bias(bias: Optional[torch.Tensor], num_heads: int, head_size: int, v_head_size: int,
                        kv_rank: int):
    """The projection-bias segments MultiHeadAttention applies ("Custom operators", section
    Microsoft MultiHeadAttention): the bias input is one vector of N*H + N*H + N*Hv values,
    the query, key and value segments in that order (the order of its size formula).  The
    query segment is always added to the query; the key and value segments are added only to
    rank-3 (packed, not yet split into heads) key and value inputs: for rank-4 key/value
    (cross-attention with pre-projected heads) only the query segment is applied.

    Returns (q_bias, k_bias, v_bias) as slices of `bias`, None where a segment is not applied."""
    if bias is None:
        return None, None, None
    nh, nhv = num_heads * head_size, num_heads * v_head_size
    if bias.dim() != 1 or bias.numel() != 2 * nh + nhv:
        raise ValueError(f"projection bias must be ({2 * nh + nhv},), got {tuple(bias.shape)}")
    if kv_rank not in (3, 4):
        raise ValueError("key/value rank must be 3 or 4")
    q_seg = bias[:nh]
    if kv_rank == 4:
        return q_seg, None, None
    return q_seg, bias[nh:2 * nh], bias[2 * nh:]


def present(past: Optional[torch.Tensor], cur: torch.Tensor, bias: Optional[torch.Tensor] = None
            ) -> torch.Tensor:
    """present = concat(past, cur [+ bias]) along the sequence axis, (B, N, P+L, D) contiguous."""
    B, N, L, D = cur.shape
    P = 0 if past is None else past.shape[2]
    keep: list = []
    out = torch.empty((B, N, P + L, D), dtype=cur.dtype)
    pv = _view(past, keep) if past is not None else _Tensor(None, 0, 0, 0, 0)
    cv = _view(cur, keep)
    rc = lib().oracle_present(_DT[cur.dtype], B, N, P, L, D, ctypes.byref(pv), ctypes.byref(cv),
                              _ptr(bias, keep), out.data_ptr())
    if rc != 0:
        raise ValueError("oracle_present rejected its arguments")
    return out


def to_double(dtype_code: int, buf: torch.Tensor) -> np.ndarray:
    """Widen every element of a 1-D CPU tensor with the oracle's own conversion."""
    buf = buf.contiguous()
    f = lib().oracle_to_double
    return np.array([f(dtype_code, buf.data_ptr(), i) for i in range(buf.numel())], dtype=np.float64)


def round_f16(x: float) -> int:
    return int(lib().oracle_round_f16(float(x)))


def round_bf16(x: float) -> int:
    return int(lib().oracle_round_bf16(float(x)))


def round_array(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """Rounds a float64 array once, to nearest even, to dtype (the oracle's own rounding)."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = torch.empty(a.shape, dtype=dtype)
    if lib().oracle_round_array(_DT[dtype], a.ctypes.data, a.size, out.data_ptr()) != 0:
        raise ValueError("oracle_round_array: dtype must be float32, float16 or bfloat16")
    return out


def gqa_rotary_positions(B: int, S: int, L: int, T: int, seqlens_k: Optional[torch.Tensor] = None):
    """Absolute positions of the rotated rows ("Microsoft GroupQueryAttention": RoPE uses
    absolute positions).  The S query rows and the L new key rows are the last rows of
    the valid sequence of Tv(b) keys, Tv(b) = seqlens_k[b] + 1 when given, else T: query
    i at Tv(b) - S + i, new key j at Tv(b) - L + j (the causal alignment's positions).
    Returns (B, S) and (B, L) int64 tensors."""
    if seqlens_k is not None:
        tv = seqlens_k.to(torch.int64).view(B, 1) + 1
    else:
        tv = torch.full((B, 1), T, dtype=torch.int64)
    return tv - S + torch.arange(S).view(1, S), tv - L + torch.arange(L).view(1, L)


def rotary(x: torch.Tensor, cos_cache: torch.Tensor, sin_cache: torch.Tensor,
           position_ids: Optional[torch.Tensor] = None, rotary_dim: int = 0,
           interleaved: bool = False) -> np.ndarray:
    """RotaryEmbedding of a (B, N, S, D) CPU view; returns float64 (B, N, S, D).

    cos_cache / sin_cache: rank-2 (max_pos, R/2) with position_ids (B, S) int64, or rank-3
    (B, S, R/2) without position ids."""
    B, N, S, D = x.shape
    keep: list = []
    xv = _view(x, keep)
    cc, sc = cos_cache.contiguous(), sin_cache.contiguous()
    keep += [cc, sc]
    ld = cc.shape[-1]
    pos_ptr, pos_sb = None, 0
    if position_ids is not None:
        pid = position_ids.to(torch.int64).contiguous()
        keep.append(pid)
        pos_ptr, pos_sb = pid.data_ptr(), pid.shape[-1] if pid.dim() == 2 else 0
    out = np.zeros((B, N, S, D), dtype=np.float64)
    rc = lib().oracle_rotary(B, N, S, D, ctypes.byref(xv), int(rotary_dim), int(bool(interleaved)),
                             cc.data_ptr(), sc.data_ptr(), _DT[cc.dtype], ld, pos_ptr, pos_sb,
                             out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_rotary rejected its arguments")
    return out
