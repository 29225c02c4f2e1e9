"""Turns a seeded workload case into the oracle's problem description (CPU tensors)."""
from __future__ import annotations

import oracle
from scaled_dot_product_gb300.workloads import Case

CAUSAL = {"none": oracle.CAUSAL_NONE, "upper_left": oracle.CAUSAL_UPPER_LEFT,
          "lower_right": oracle.CAUSAL_LOWER_RIGHT}
KEEP = {"none": oracle.KEEP_NONE, "bool": oracle.KEEP_BOOL, "filter": oracle.KEEP_FILTER}
LENS = {"none": oracle.LEN_NONE, "nonpad": oracle.LEN_NONPAD_I64,
        "keylen": oracle.LEN_KEYLEN_I32, "seqlens_k": oracle.LEN_SEQLENS_K_I32}


def _expand(m, case: Case):
    if m is None:
        return None
    return m.expand(case.B, case.Nq, case.S, m.shape[-1])


def rotated_qk(c: Case):
    """(q, k) after GroupQueryAttention's rotary step, each rounded once to the case's
    dtype (RotaryEmbedding's output has the input's element type); unchanged without it."""
    q, k, v = c.views()
    if c.rotary_cos is None:
        return q, k
    qpos, kpos = oracle.gqa_rotary_positions(
        c.B, c.S, c.L, c.T, c.lens if c.len_kind == "seqlens_k" else None)
    rq = oracle.rotary(q, c.rotary_cos, c.rotary_sin, qpos, c.rotary_dim, c.rotary_interleaved)
    rk = oracle.rotary(k, c.rotary_cos, c.rotary_sin, kpos, c.rotary_dim, c.rotary_interleaved)
    return oracle.round_array(rq, c.dtype), oracle.round_array(rk, c.dtype)


def problem(case: Case) -> oracle.Problem:
    c = case.to("cpu")
    _, _, v = c.views()
    q, k = rotated_qk(c)
    return oracle.Problem(
        q=q, k=k, v=v, past_k=c.past_k, past_v=c.past_v,
        q_bias=c.q_bias, k_bias=c.k_bias, v_bias=c.v_bias,
        scale=c.scale, softcap=c.softcap, causal=CAUSAL[c.causal], window=c.window,
        head_sink=c.head_sink, add_mask=_expand(c.add_mask, c), keep_mask=_expand(c.keep_mask, c),
        keep_kind=KEEP[c.keep_kind], len_kind=LENS[c.len_kind], lens=c.lens,
        mask_filter_value=c.mask_filter_value, softcap_before_bias=c.softcap_before_bias)


def expected_present(case: Case):
    """(present_k, present_v) from the oracle, or (None, None) when the case wants none."""
    if not case.want_present:
        return None, None
    c = case.to("cpu")
    _, _, v = c.views()
    _, k = rotated_qk(c)
    return oracle.present(c.past_k, k, c.k_bias), oracle.present(c.past_v, v, c.v_bias)
