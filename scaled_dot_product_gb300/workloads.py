"""Seeded synthetic workloads for scaled dot-product attention.

This module only draws inputs and describes their layout: it holds none of the method's
arithmetic, imports neither the CUDA binding nor the oracle, and is the one piece shared
by the parity tests, the benchmark and the smoke check.

Recipe: values are drawn in float32 from ``torch.Generator().manual_seed(seed)`` on the
CPU (chunked for large tensors, so memory stays bounded and the stream is fixed), then
rounded once, round-to-nearest-even, to the case's dtype.  The default seed of a named
workload is 1000 + its index (1..5).

Layouts follow the operator contracts: "bsnh" is the packed rank-3 layout (B, S, N*H),
"bnsh" the rank-4 layout (B, N, S, H).  ``as4d`` turns either into a (B, N, S, H) view
without copying.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

_CHUNK = 1 << 24


def _normal(gen: torch.Generator, shape, dtype, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        x = torch.randn(n, generator=gen, dtype=torch.float32)
        if std != 1.0 or mean != 0.0:
            x = x * std + mean
        flat[s:s + n] = x.to(dtype)
    return out


def _uniform(gen: torch.Generator, shape, dtype, lo: float, hi: float) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    for s in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - s)
        x = torch.rand(n, generator=gen, dtype=torch.float32) * (hi - lo) + lo
        flat[s:s + n] = x.to(dtype)
    return out


def _randint(gen: torch.Generator, n: int, lo: int, hi_inclusive: int, dtype) -> torch.Tensor:
    return torch.randint(lo, hi_inclusive + 1, (n,), generator=gen, dtype=torch.int64).to(dtype)


def rope_caches(max_pos: int, half: int, dtype, base: float = 10000.0):
    """cos / sin input tables (max_pos, half) of RoFormer's angle schedule
    pos * base^(-d/half), computed in float64 and converted to dtype by torch."""
    pos = torch.arange(max_pos, dtype=torch.float64).view(-1, 1)
    inv = base ** (-torch.arange(half, dtype=torch.float64) / half)
    ang = pos * inv.view(1, -1)
    return torch.cos(ang).to(dtype).contiguous(), torch.sin(ang).to(dtype).contiguous()


def as4d(t: Optional[torch.Tensor], layout: str, n_heads: int) -> Optional[torch.Tensor]:
    """(B, N, S, D) view of a tensor stored as rank-3 (B, S, N*D) or rank-4 (B, N, S, D)."""
    if t is None:
        return None
    if layout == "bnsh":
        assert t.dim() == 4
        return t
    assert layout == "bsnh" and t.dim() == 3 and t.shape[2] % n_heads == 0
    B, S, ND = t.shape
    return t.view(B, S, n_heads, ND // n_heads).permute(0, 2, 1, 3)


@dataclass
class Case:
    """One attention problem in operator terms (tensors on the CPU until moved)."""
    name: str
    dtype: torch.dtype
    B: int
    Nq: int
    Nkv: int
    S: int
    L: int
    P: int
    H: int
    Hv: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_layout: str = "bnsh"
    kv_layout: str = "bnsh"
    past_k: Optional[torch.Tensor] = None          # (B, Nkv, P, H)
    past_v: Optional[torch.Tensor] = None
    want_present: bool = False
    q_bias: Optional[torch.Tensor] = None          # (Nq*H,)
    k_bias: Optional[torch.Tensor] = None          # (Nkv*H,)
    v_bias: Optional[torch.Tensor] = None          # (Nkv*Hv,)
    proj_bias: Optional[torch.Tensor] = None       # MHA (2*N*H + N*Hv,) as the operator receives it
    scale: Optional[float] = None
    softcap: float = 0.0
    causal: str = "none"                           # none | upper_left | lower_right
    window: int = -1
    head_sink: Optional[torch.Tensor] = None       # (Nq,)
    add_mask: Optional[torch.Tensor] = None        # 4-D, broadcastable to (B, Nq, S, Tm)
    keep_mask: Optional[torch.Tensor] = None       # 4-D, broadcastable to (B, Nq, S, Tm)
    keep_kind: str = "none"                        # none | bool | filter
    lens: Optional[torch.Tensor] = None            # (B,)
    len_kind: str = "none"                         # none | nonpad | keylen | seqlens_k
    mask_filter_value: float = -10000.0
    softcap_before_bias: bool = False
    rotary_cos: Optional[torch.Tensor] = None      # (max_pos, R/2), dtype of q
    rotary_sin: Optional[torch.Tensor] = None
    rotary_dim: int = 0                            # R; 0 means H
    rotary_interleaved: bool = False
    seed: int = 0
    notes: Dict[str, str] = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.P + self.L

    def views(self):
        """(q, k, v) as (B, N, S, D) views of the stored tensors."""
        return (as4d(self.q, self.q_layout, self.Nq), as4d(self.k, self.kv_layout, self.Nkv),
                as4d(self.v, self.kv_layout, self.Nkv))

    def y_shape(self):
        if self.q_layout == "bsnh":
            return (self.B, self.S, self.Nq * self.Hv)
        return (self.B, self.Nq, self.S, self.Hv)

    def to(self, device) -> "Case":
        """Same case with every tensor moved (strides of the stored tensors are kept)."""
        kw = {}
        for f in dataclasses.fields(self):
            val = getattr(self, f.name)
            kw[f.name] = val.to(device) if isinstance(val, torch.Tensor) else val
        return Case(**kw)

    def input_bytes(self) -> int:
        n = 0
        for f in dataclasses.fields(self):
            val = getattr(self, f.name)
            if isinstance(val, torch.Tensor) and f.name != "proj_bias":
                n += val.numel() * val.element_size()
        return n


def make_case(name: str, *, dtype=torch.bfloat16, B=1, Nq=2, Nkv=None, S=16, L=None, P=0, H=8,
              Hv=None, q_layout="bnsh", kv_layout="bnsh", seed=0, want_present=False,
              scale=None, softcap=0.0, causal="none", window=-1, sink=False,
              add_mask=None, add_mask_shape=None, add_mask_range=(-1.0, 0.0),
              keep_kind="none", keep_mask_shape=None, keep_density=0.8,
              len_kind="none", len_range=None, qkv_bias=None, proj_bias_std=0.02,
              mask_filter_value=-10000.0, softcap_before_bias=False, rotary=None, rotary_dim=0,
              rotary_max_pos=None, rotary_base=10000.0) -> Case:
    """Draw a case.  Draw order is fixed: q, k, v, past_k, past_v, biases, sink, masks, lens.

    add_mask: None | "float" (uniform in add_mask_range, dtype of q, shape add_mask_shape).
    keep_kind: "bool" draws a u8 keep mask, "filter" an int32 one, both with P(keep)=keep_density
    and shape keep_mask_shape.  len_range: (lo, hi) inclusive for the per-batch lengths.
    qkv_bias: None | "q" | "qkv" (MHA projection-bias segments drawn N(0, proj_bias_std)).
    rotary: None | "half" | "interleaved": rank-2 cos/sin caches of rotary_max_pos rows
    (default P + L) for R = rotary_dim (0: H) channels (no random draw; see rope_caches).
    """
    Nkv = Nq if Nkv is None else Nkv
    L = S if L is None else L
    Hv = H if Hv is None else Hv
    gen = torch.Generator().manual_seed(seed)
    if q_layout == "bsnh":
        q = _normal(gen, (B, S, Nq * H), dtype)
    else:
        q = _normal(gen, (B, Nq, S, H), dtype)
    if kv_layout == "bsnh":
        k = _normal(gen, (B, L, Nkv * H), dtype)
        v = _normal(gen, (B, L, Nkv * Hv), dtype)
    else:
        k = _normal(gen, (B, Nkv, L, H), dtype)
        v = _normal(gen, (B, Nkv, L, Hv), dtype)
    past_k = past_v = None
    if P > 0:
        past_k = _normal(gen, (B, Nkv, P, H), dtype)
        past_v = _normal(gen, (B, Nkv, P, Hv), dtype)
    q_bias = k_bias = v_bias = proj = None
    if qkv_bias is not None:
        proj = _normal(gen, (Nq * H + Nkv * H + Nkv * Hv,), dtype, std=proj_bias_std)
        q_bias = proj[: Nq * H]
        if qkv_bias == "qkv":
            k_bias = proj[Nq * H: Nq * H + Nkv * H]
            v_bias = proj[Nq * H + Nkv * H:]
    head_sink = _normal(gen, (Nq,), dtype) if sink else None
    T = P + L
    am = None
    if add_mask == "float":
        shape = add_mask_shape or (B, Nq, S, T)
        am = _uniform(gen, shape, dtype, *add_mask_range)
    km = None
    if keep_kind != "none":
        shape = keep_mask_shape or (B, 1, S, T)
        draw = torch.rand(shape, generator=gen) < keep_density
        km = draw.to(torch.uint8 if keep_kind == "bool" else torch.int32)
    lens = None
    if len_kind != "none":
        lo, hi = len_range
        ldt = torch.int64 if len_kind == "nonpad" else torch.int32
        lens = _randint(gen, B, lo, hi, ldt)
    rc = rs = None
    if rotary is not None:
        R = rotary_dim or H
        rc, rs = rope_caches(rotary_max_pos or T, R // 2, dtype, rotary_base)
    return Case(name=name, dtype=dtype, B=B, Nq=Nq, Nkv=Nkv, S=S, L=L, P=P, H=H, Hv=Hv,
                q=q, k=k, v=v, q_layout=q_layout, kv_layout=kv_layout, past_k=past_k,
                past_v=past_v, want_present=want_present, q_bias=q_bias, k_bias=k_bias,
                v_bias=v_bias, proj_bias=proj, scale=scale, softcap=softcap, causal=causal,
                window=window, head_sink=head_sink, add_mask=am, keep_mask=km,
                keep_kind=keep_kind, lens=lens, len_kind=len_kind,
                mask_filter_value=mask_filter_value, softcap_before_bias=softcap_before_bias,
                rotary_cos=rc, rotary_sin=rs, rotary_dim=rotary_dim,
                rotary_interleaved=rotary == "interleaved", seed=seed)


def draw_dy(case: Case, seed: int) -> torch.Tensor:
    """Upstream gradient dY for the backward, in y's layout (rank-3 when the query is
    packed): N(0, 1) drawn in fp32 from its own seeded generator, rounded once to the dtype."""
    gen = torch.Generator().manual_seed(seed)
    return _normal(gen, case.y_shape(), case.dtype)


@dataclass
class RotaryInputs:
    """Inputs of one standalone RotaryEmbedding call."""
    x: torch.Tensor                      # (B, N, S, D) or packed (B, S, N*D)
    layout: str                          # "bnsh" | "bsnh"
    N: int
    cos: torch.Tensor                    # (max_pos, R/2) or (B, S, R/2)
    sin: torch.Tensor
    position_ids: Optional[torch.Tensor]  # (B, S) int64, or None with rank-3 caches
    rotary_dim: int
    interleaved: bool

    def to(self, device) -> "RotaryInputs":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, x=mv(self.x), cos=mv(self.cos), sin=mv(self.sin),
                                   position_ids=mv(self.position_ids))


def make_rotary_inputs(*, B=2, N=3, S=17, D=64, dtype=torch.bfloat16, layout="bnsh", rotary_dim=0,
                       interleaved=False, cache="ids", max_pos=None, seed=0) -> RotaryInputs:
    """x ~ N(0, 1); cache "ids": rank-2 tables of max_pos rows (default 2*S + 5) and position
    ids drawn uniformly in [0, max_pos); cache "per_token": rank-3 (B, S, R/2) tables."""
    gen = torch.Generator().manual_seed(seed)
    x = _normal(gen, (B, S, N * D) if layout == "bsnh" else (B, N, S, D), dtype)
    half = (rotary_dim or D) // 2
    if cache == "ids":
        mp = max_pos or 2 * S + 5
        cos, sin = rope_caches(mp, half, dtype)
        pid = torch.randint(0, mp, (B, S), generator=gen, dtype=torch.int64)
    else:
        cos, sin = rope_caches(B * S, half, dtype)
        cos, sin = cos.view(B, S, half), sin.view(B, S, half)
        pid = None
    return RotaryInputs(x=x, layout=layout, N=N, cos=cos, sin=sin, position_ids=pid,
                        rotary_dim=rotary_dim, interleaved=interleaved)


# ----------------------------------------------------------------------------------------
# The five named workloads.  Index 1..5; the small variants keep every feature and the
# layout but shrink the sizes so the oracle finishes in seconds while still spanning
# several 128-row tiles and a ragged tail.
# ----------------------------------------------------------------------------------------

WORKLOADS = {
    1: "attention_f32_b1_n2_s16_h8",
    2: "attention_gqa_bf16_b2_s2048_q32_kv8_h128_causal_softcap30_nonpad",
    3: "gqa_bf16_b1_s4096_q64_kv8_h64_window1024_sink",
    4: "mha_decode_f16_b64_n32_h128_past4095_keylen",
    5: "mha_cross_f16_b8_s448_n20_h64_kv1500_bias",
    # not a headline configuration: measures MultiHeadAttention's binary key mask and
    # unidirectional (lower-right causal) rule on the tensor-core path
    6: "mha_prefill_f16_b4_s2048_n16_h128_binary_mask_unidirectional",
}


def workload(idx: int, small: bool = False, seed: Optional[int] = None, batch: Optional[int] = None) -> Case:
    """Named workload idx (1..5); `batch` overrides the batch size (for profiling captures
    that must stay small)."""
    seed = 1000 + idx if seed is None else seed
    name = WORKLOADS[idx] + ("_small" if small else "")
    if idx == 1:
        return make_case(name, dtype=torch.float32, B=1, Nq=2, S=16, H=8, seed=seed)
    if idx == 2:
        B, S, Nq, Nkv, H = (2, 300, 8, 2, 128) if small else (2, 2048, 32, 8, 128)
        B = batch if batch is not None else B
        return make_case(name, dtype=torch.bfloat16, B=B, Nq=Nq, Nkv=Nkv, S=S, H=H,
                         q_layout="bsnh", kv_layout="bsnh", seed=seed, causal="upper_left",
                         softcap=30.0, len_kind="nonpad", len_range=(S // 2, S))
    if idx == 3:
        B, S, Nq, Nkv, H, W = (1, 400, 16, 2, 64, 100) if small else (1, 4096, 64, 8, 64, 1024)
        c = make_case(name, dtype=torch.bfloat16, B=B, Nq=Nq, Nkv=Nkv, S=S, H=H,
                      q_layout="bsnh", kv_layout="bsnh", seed=seed, causal="lower_right",
                      window=W, sink=True)
        c.lens = torch.full((B,), S - 1, dtype=torch.int32)     # seqlens_k = total - 1
        c.len_kind = "seqlens_k"
        return c
    if idx == 4:
        B, N, P, H = (4, 4, 700, 128) if small else (64, 32, 4095, 128)
        B = batch if batch is not None else B
        return make_case(name, dtype=torch.float16, B=B, Nq=N, S=1, L=1, P=P, H=H,
                         q_layout="bsnh", kv_layout="bsnh", seed=seed, want_present=True,
                         len_kind="keylen", len_range=((P + 1) // 4, P + 1))
    if idx == 5:
        B, S, N, H, Lk = (2, 200, 4, 64, 333) if small else (8, 448, 20, 64, 1500)
        return make_case(name, dtype=torch.float16, B=B, Nq=N, S=S, L=Lk, H=H,
                         q_layout="bsnh", kv_layout="bnsh", seed=seed, qkv_bias="q",
                         add_mask="float", add_mask_shape=(B, 1, S, Lk), add_mask_range=(-1.0, 0.0))
    if idx == 6:
        B, S, N, H = (2, 300, 4, 128) if small else (4, 2048, 16, 128)
        B = batch if batch is not None else B
        return make_case(name, dtype=torch.float16, B=B, Nq=N, S=S, H=H, q_layout="bsnh", kv_layout="bsnh",
                         seed=seed, causal="lower_right", keep_kind="filter", keep_mask_shape=(B, 1, S, S),
                         keep_density=0.9)
    raise KeyError(idx)


def all_workloads(small: bool = True) -> List[Case]:
    return [workload(i, small=small) for i in sorted(WORKLOADS)]
