"""Pins of the double-precision oracle to facts outside itself (CPU only).

Each test checks the oracle against one of: a library routine on a special case
(torch float64 scaled_dot_product_attention, numpy / torch dtype conversions), a
closed form, an invariant the operator contracts fix, or an example stated on the
documentation pages (tests/golden/contract_examples.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
from oracle import Problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "contract_examples.json")


def rnd(*shape, seed=0, dtype=torch.float64, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * std).to(dtype)


def run(q, k, v, **kw):
    return oracle.attention(Problem(q=q, k=k, v=v, **kw))


def sdpa(q, k, v, **kw):
    return F.scaled_dot_product_attention(q.double(), k.double(), v.double(), **kw).numpy()


# ---------------------------------------------------------------- element conversions

def test_f16_widening_all_bit_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    got = oracle.to_double(oracle.F16, bits.view(torch.float16))
    want = bits.numpy().view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_bf16_widening_all_bit_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    got = oracle.to_double(oracle.BF16, bits.view(torch.bfloat16))
    want = bits.view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def _rounding_samples():
    g = np.random.default_rng(7)
    mags = np.concatenate([
        g.standard_normal(20000),
        g.standard_normal(5000) * 1e-6,       # f16 subnormal range
        g.standard_normal(5000) * 1e4,        # near the f16 overflow
        g.standard_normal(2000) * 1e-40,      # binary32/bf16 subnormal range
        g.standard_normal(2000) * 1e38,
    ])
    with np.errstate(over="ignore"):
        mags = mags.astype(np.float32)
    # exact ties between two neighbouring f16 / bf16 values
    base16 = g.standard_normal(3000).astype(np.float16).astype(np.float32)
    ties16 = (base16 + np.spacing(base16.astype(np.float16)).astype(np.float32) / 2).astype(np.float32)
    return np.concatenate([mags, ties16, np.float32([0.0, -0.0, 65504, 65519, 65520, 65536, 1e-8])])


def test_f16_rounding_matches_numpy():
    xs = _rounding_samples()
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.round_f16(float(x)) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_bf16_rounding_matches_torch():
    xs = _rounding_samples()
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_bf16(float(x)) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_array_rounding_is_one_rounding_from_double():
    """round_array rounds doubles once: it matches numpy's direct double->half conversion
    and the scalar (pinned) roundings, and does not round through float32 first."""
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 5, 4000),
                         _rounding_samples().astype(np.float64)])
    with np.errstate(over="ignore"):
        np.testing.assert_array_equal(oracle.round_array(xs, torch.float16).view(torch.int16).numpy(),
                                      xs.astype(np.float16).view(np.int16))
    got = oracle.round_array(xs, torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, np.array([oracle.round_bf16(x) for x in xs], dtype=np.uint16))
    np.testing.assert_array_equal(oracle.round_array(xs, torch.float32).numpy(), xs.astype(np.float32))
    # just above a bf16 tie by less than a float32 ulp: a float32 detour would round to even (down)
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert float(oracle.round_array(np.array([x]), torch.bfloat16)[0]) == 1.0 + 2.0 ** -7
    x = 1.0 + 2.0 ** -11 + 2.0 ** -40                     # same for float16
    assert float(oracle.round_array(np.array([x]), torch.float16)[0]) == 1.0 + 2.0 ** -10


# ---------------------------------------------------------------- library special cases

@pytest.mark.parametrize("shape", [(1, 2, 16, 16, 8), (2, 3, 5, 9, 16), (1, 1, 1, 7, 4)])
def test_plain_attention_equals_torch_sdpa(shape):
    B, N, S, T, H = shape
    q, k, v = rnd(B, N, S, H, seed=1), rnd(B, N, T, H, seed=2), rnd(B, N, T, H, seed=3)
    np.testing.assert_allclose(run(q, k, v), sdpa(q, k, v), rtol=0, atol=1e-12)


def test_explicit_scale_and_value_width():
    q, k, v = rnd(2, 2, 6, 8, seed=4), rnd(2, 2, 9, 8, seed=5), rnd(2, 2, 9, 5, seed=6)
    np.testing.assert_allclose(run(q, k, v, scale=0.37), sdpa(q, k, v, scale=0.37), atol=1e-12)


@pytest.mark.parametrize("S,T", [(7, 7), (4, 9), (9, 4)])
def test_upper_left_causal_equals_torch_is_causal(S, T):
    q, k, v = rnd(1, 2, S, 8, seed=7), rnd(1, 2, T, 8, seed=8), rnd(1, 2, T, 8, seed=9)
    got = run(q, k, v, causal=oracle.CAUSAL_UPPER_LEFT)
    want = sdpa(q, k, v, is_causal=True)
    rows_ok = np.isfinite(want).all(axis=-1)            # torch gives NaN on empty rows
    np.testing.assert_allclose(got[rows_ok], want[rows_ok], atol=1e-12)
    np.testing.assert_array_equal(got[~rows_ok], 0.0)     # reading: empty row -> zeros


def test_lower_right_causal_with_past_equals_torch_causal_lower_right():
    B, N, S, P, H = 2, 2, 3, 5, 8
    q = rnd(B, N, S, H, seed=10)
    past_k, past_v = rnd(B, N, P, H, seed=11), rnd(B, N, P, H, seed=12)
    k, v = rnd(B, N, S, H, seed=13), rnd(B, N, S, H, seed=14)
    got = run(q, k, v, past_k=past_k, past_v=past_v, causal=oracle.CAUSAL_LOWER_RIGHT)
    kt, vt = torch.cat([past_k, k], 2), torch.cat([past_v, v], 2)
    want = sdpa(q, kt, vt, attn_mask=causal_lower_right(S, P + S))
    np.testing.assert_allclose(got, want, atol=1e-12)


def test_bool_and_float_masks_equal_torch():
    B, N, S, T, H = 2, 3, 5, 7, 8
    q, k, v = rnd(B, N, S, H, seed=15), rnd(B, N, T, H, seed=16), rnd(B, N, T, H, seed=17)
    g = torch.Generator().manual_seed(18)
    keep = torch.rand(B, 1, S, T, generator=g) < 0.7
    keep[..., 0] = True
    got = run(q, k, v, keep_mask=keep.to(torch.uint8).expand(B, N, S, T), keep_kind=oracle.KEEP_BOOL)
    np.testing.assert_allclose(got, sdpa(q, k, v, attn_mask=keep), atol=1e-12)
    fm = rnd(1, N, S, T, seed=19)
    got = run(q, k, v, add_mask=fm.expand(B, N, S, T))
    np.testing.assert_allclose(got, sdpa(q, k, v, attn_mask=fm), atol=1e-12)


def test_grouped_heads_equal_torch_enable_gqa():
    B, Nq, Nkv, S, T, H = 2, 8, 2, 5, 6, 16
    q, k, v = rnd(B, Nq, S, H, seed=20), rnd(B, Nkv, T, H, seed=21), rnd(B, Nkv, T, H, seed=22)
    np.testing.assert_allclose(run(q, k, v), sdpa(q, k, v, enable_gqa=True), atol=1e-12)


@pytest.mark.parametrize("kind", ["nonpad", "keylen", "seqlens_k"])
def test_length_vectors_equal_sliced_torch(kind):
    B, N, S, T, H = 3, 2, 4, 10, 8
    q, k, v = rnd(B, N, S, H, seed=23), rnd(B, N, T, H, seed=24), rnd(B, N, T, H, seed=25)
    n = [1, 6, 10]
    if kind == "nonpad":
        lens, code = torch.tensor(n, dtype=torch.int64), oracle.LEN_NONPAD_I64
    elif kind == "keylen":
        lens, code = torch.tensor(n, dtype=torch.int32), oracle.LEN_KEYLEN_I32
    else:
        lens, code = torch.tensor([x - 1 for x in n], dtype=torch.int32), oracle.LEN_SEQLENS_K_I32
    got = run(q, k, v, lens=lens, len_kind=code)
    for b in range(B):
        want = sdpa(q[b:b + 1], k[b:b + 1, :, :n[b]], v[b:b + 1, :, :n[b]])
        np.testing.assert_allclose(got[b:b + 1], want, atol=1e-12)


def test_projection_bias_segments_equal_torch_on_biased_inputs():
    B, N, S, T, H, Hv = 2, 2, 4, 6, 8, 4
    q, k, v = rnd(B, N, S, H, seed=26), rnd(B, N, T, H, seed=27), rnd(B, N, T, Hv, seed=28)
    bias = rnd(2 * N * H + N * Hv, seed=29)
    qb, kb, vb = bias[:N * H], bias[N * H:2 * N * H], bias[2 * N * H:]
    got = run(q, k, v, q_bias=qb, k_bias=kb, v_bias=vb)
    want = sdpa(q + qb.view(1, N, 1, H), k + kb.view(1, N, 1, H), v + vb.view(1, N, 1, Hv))
    np.testing.assert_allclose(got, want, atol=1e-12)


# ---------------------------------------------------------------- present outputs

def test_present_holds_past_then_new_bit_exact():
    cases = json.load(open(GOLDEN))["present_positions"]["cases"]
    for c in cases:
        P, L = c["P"] if c["P"] < 100 else 9, c["L"]
        past = rnd(2, 3, P, 8, seed=30, dtype=torch.float16) if P else None
        cur = rnd(2, 3, L, 8, seed=31, dtype=torch.float16)
        pres = oracle.present(past, cur)
        assert pres.shape[2] == P + L
        if P:
            assert torch.equal(pres[:, :, :P].view(torch.int16), past.view(torch.int16))
        assert torch.equal(pres[:, :, P:].view(torch.int16), cur.view(torch.int16))


def test_present_with_bias_rounds_once():
    cur = rnd(2, 3, 5, 8, seed=32, dtype=torch.float16)
    bias = rnd(3 * 8, seed=33, dtype=torch.float16, std=0.02)
    pres = oracle.present(None, cur, bias)
    exact = cur.double().numpy() + bias.double().numpy().reshape(1, 3, 1, 8)
    want = exact.astype(np.float16)                      # numpy rounds float64 -> float16 once
    np.testing.assert_array_equal(pres.numpy().view(np.uint16), want.view(np.uint16))
    curb = rnd(2, 3, 5, 8, seed=34, dtype=torch.bfloat16)
    biasb = rnd(3 * 8, seed=35, dtype=torch.bfloat16, std=0.02)
    presb = oracle.present(None, curb, biasb)
    sum32 = curb.float() + biasb.float().view(1, 3, 1, 8)  # exact in binary32 at these magnitudes
    assert torch.equal(sum32.double(), curb.double() + biasb.double().view(1, 3, 1, 8))
    assert torch.equal(presb.view(torch.int16), sum32.to(torch.bfloat16).view(torch.int16))


# ---------------------------------------------------------------- closed forms

def test_identical_keys_give_mean_of_admitted_values():
    B, N, S, T, H, Hv = 2, 2, 6, 11, 8, 3
    q = rnd(B, N, S, H, seed=36)
    k = rnd(1, 1, 1, H, seed=37).expand(B, N, T, H).contiguous()
    v = rnd(B, N, T, Hv, seed=38)
    lens = torch.tensor([7, 11], dtype=torch.int64)
    got = run(q, k, v, causal=oracle.CAUSAL_LOWER_RIGHT, window=3,
              lens=lens, len_kind=oracle.LEN_NONPAD_I64)
    for b in range(B):
        for i in range(S):
            pos = T - S + i
            adm = [j for j in range(T) if j <= pos and j >= pos - 2 and j < lens[b]]
            want = v[b, :, adm].mean(dim=1).numpy() if adm else np.zeros((N, Hv))
            np.testing.assert_allclose(got[b, :, i], want, atol=1e-12)


def test_window_example_from_the_pages():
    ex = json.load(open(GOLDEN))["local_window_example"]
    W, before = ex["local_window_size"], ex["preceding_positions_attended"]
    T = W + 52
    q = torch.zeros(1, 1, T, 1, dtype=torch.float64)
    k = torch.zeros(1, 1, T, 1, dtype=torch.float64)
    v = torch.arange(T, dtype=torch.float64).view(1, 1, T, 1)
    got = run(q, k, v, causal=oracle.CAUSAL_UPPER_LEFT, window=W)
    for i in (0, 100, W - 1, W, T - 1):
        lo = max(0, i - before)
        assert got[0, 0, i, 0] == pytest.approx((lo + i) / 2, abs=1e-9)


def test_window_of_one_returns_the_current_value():
    q, k, v = rnd(1, 2, 5, 8, seed=39), rnd(1, 2, 9, 8, seed=40), rnd(1, 2, 9, 4, seed=41)
    got = run(q, k, v, causal=oracle.CAUSAL_LOWER_RIGHT, window=1)
    for i in range(5):
        np.testing.assert_allclose(got[0, :, i], v[0, :, 4 + i].numpy(), atol=1e-12)


def test_single_admitted_key_returns_its_value():
    q, k, v = rnd(2, 2, 3, 8, seed=42), rnd(2, 2, 6, 8, seed=43), rnd(2, 2, 6, 5, seed=44)
    got = run(q, k, v, lens=torch.tensor([1, 1], dtype=torch.int64), len_kind=oracle.LEN_NONPAD_I64)
    np.testing.assert_allclose(got, v[:, :, :1].expand(2, 2, 3, 5).numpy(), atol=1e-12)


def test_head_sink_closed_form():
    # n admitted keys, all scores 0, values 1: y = n / (n + e^sink); sink = ln n gives 1/2.
    n, T = 6, 9
    q = torch.zeros(1, 3, 1, 4, dtype=torch.float64)
    k = torch.zeros(1, 3, T, 4, dtype=torch.float64)
    v = torch.ones(1, 3, T, 1, dtype=torch.float64)
    sink = torch.tensor([math.log(n), 0.0, 2.5], dtype=torch.float64)
    got = run(q, k, v, head_sink=sink, lens=torch.tensor([n], dtype=torch.int64),
              len_kind=oracle.LEN_NONPAD_I64)
    assert got[0, 0, 0, 0] == pytest.approx(0.5, abs=1e-14)
    assert got[0, 1, 0, 0] == pytest.approx(n / (n + 1.0), abs=1e-14)
    assert got[0, 2, 0, 0] == pytest.approx(n / (n + math.exp(2.5)), abs=1e-14)


def _softcap_two_keys(add_first=0.0, raw_first=None, **kw):
    # c = 2 ln 3 and a raw score c*atanh(1/2) = (ln 3)^2 cap to c/2 = ln 3: weights 3/4, 1/4.
    c = 2 * math.log(3.0)
    raw = (math.log(3.0) ** 2) if raw_first is None else raw_first
    q = torch.ones(1, 1, 1, 1, dtype=torch.float64)
    k = torch.tensor([raw, 0.0], dtype=torch.float64).view(1, 1, 2, 1)
    v = torch.tensor([1.0, 0.0], dtype=torch.float64).view(1, 1, 2, 1)
    mask = torch.tensor([add_first, 0.0], dtype=torch.float64).view(1, 1, 1, 2)
    return run(q, k, v, scale=1.0, softcap=c, add_mask=mask, **kw)[0, 0, 0, 0], c


def test_softcap_closed_form():
    y, _ = _softcap_two_keys()
    assert y == pytest.approx(0.75, abs=1e-14)


def test_bias_enters_before_softcap_in_the_stage_order():
    # raw score 0 with a finite bias (ln 3)^2: bias-then-cap gives ln 3 -> 3/4;
    # cap-then-bias gives (ln 3)^2 -> e^{(ln3)^2} / (1 + e^{(ln3)^2}).
    b = math.log(3.0) ** 2
    y, _ = _softcap_two_keys(add_first=b, raw_first=0.0)
    assert y == pytest.approx(0.75, abs=1e-14)
    y2, _ = _softcap_two_keys(add_first=b, raw_first=0.0, softcap_before_bias=True)
    assert y2 == pytest.approx(math.exp(b) / (1 + math.exp(b)), abs=1e-14)


def test_negative_infinite_mask_entry_stays_excluded_under_softcap():
    y, _ = _softcap_two_keys(add_first=-math.inf)
    assert y == 0.0


# ---------------------------------------------------------------- invariants

def test_gqa_equals_mha_with_repeated_kv_heads():
    B, Nq, Nkv, S, T, H = 2, 6, 3, 5, 8, 8
    q, k, v = rnd(B, Nq, S, H, seed=45), rnd(B, Nkv, T, H, seed=46), rnd(B, Nkv, T, H, seed=47)
    sink = rnd(Nq, seed=48)
    kw = dict(causal=oracle.CAUSAL_LOWER_RIGHT, window=4, head_sink=sink, softcap=3.0)
    g = Nq // Nkv
    a = run(q, k, v, **kw)
    b = run(q, k.repeat_interleave(g, 1), v.repeat_interleave(g, 1), **kw)
    np.testing.assert_allclose(a, b, atol=0)


def test_window_wider_than_sequence_equals_full_causal():
    q, k, v = rnd(1, 2, 7, 8, seed=49), rnd(1, 2, 7, 8, seed=50), rnd(1, 2, 7, 8, seed=51)
    for causal in (oracle.CAUSAL_UPPER_LEFT, oracle.CAUSAL_LOWER_RIGHT):
        a = run(q, k, v, causal=causal, window=7)
        b = run(q, k, v, causal=causal, window=1 << 30)
        c = run(q, k, v, causal=causal)
        np.testing.assert_array_equal(a, c)
        np.testing.assert_array_equal(b, c)


def test_sink_minus_infinity_is_no_sink_and_large_sink_drives_output_to_zero():
    q, k, v = rnd(1, 2, 4, 8, seed=52), rnd(1, 2, 6, 8, seed=53), rnd(1, 2, 6, 8, seed=54)
    none = run(q, k, v)
    ninf = run(q, k, v, head_sink=torch.full((2,), -math.inf, dtype=torch.float64))
    np.testing.assert_array_equal(none, ninf)
    big = run(q, k, v, head_sink=torch.full((2,), 200.0, dtype=torch.float64))
    assert np.abs(big).max() < 1e-60
    mid = run(q, k, v, head_sink=torch.full((2,), 0.5, dtype=torch.float64))
    assert (np.abs(mid) < np.abs(none) + 1e-15).all()    # weights sum below one, same direction


def test_softcap_zero_is_off_and_huge_softcap_converges():
    q, k, v = rnd(1, 2, 4, 8, seed=55), rnd(1, 2, 6, 8, seed=56), rnd(1, 2, 6, 8, seed=57)
    off = run(q, k, v)
    np.testing.assert_array_equal(run(q, k, v, softcap=0.0), off)
    np.testing.assert_allclose(run(q, k, v, softcap=1e7), off, atol=1e-10)
    capped = run(q, k, v, softcap=0.5)
    assert np.abs(capped - off).max() > 1e-3


def test_trivial_masks_are_no_ops_and_short_masks_are_padded():
    B, N, S, T, H = 1, 2, 4, 7, 8
    q, k, v = rnd(B, N, S, H, seed=58), rnd(B, N, T, H, seed=59), rnd(B, N, T, H, seed=60)
    base = run(q, k, v)
    ones = torch.ones(B, N, S, T, dtype=torch.uint8)
    np.testing.assert_array_equal(run(q, k, v, keep_mask=ones, keep_kind=oracle.KEEP_BOOL), base)
    np.testing.assert_array_equal(run(q, k, v, add_mask=torch.zeros(B, N, S, T, dtype=torch.float64)), base)
    const = torch.full((B, N, S, T), -3.25, dtype=torch.float64)
    np.testing.assert_allclose(run(q, k, v, add_mask=const), base, atol=1e-13)
    # a mask of width 5 < T behaves like a full-width mask padded with false / -inf
    short = (torch.rand(B, N, S, 5, generator=torch.Generator().manual_seed(61)) < 0.8).to(torch.uint8)
    short[..., 0] = 1
    padded = torch.zeros(B, N, S, T, dtype=torch.uint8)
    padded[..., :5] = short
    np.testing.assert_array_equal(run(q, k, v, keep_mask=short, keep_kind=oracle.KEEP_BOOL),
                                  run(q, k, v, keep_mask=padded, keep_kind=oracle.KEEP_BOOL))
    fshort = rnd(B, N, S, 5, seed=62)
    fpad = torch.full((B, N, S, T), -math.inf, dtype=torch.float64)
    fpad[..., :5] = fshort
    np.testing.assert_array_equal(run(q, k, v, add_mask=fshort), run(q, k, v, add_mask=fpad))


def test_binary_filter_mask_equals_key_lengths_and_uses_the_filter_value():
    B, N, S, T, H = 2, 2, 3, 8, 8
    q, k, v = rnd(B, N, S, H, seed=63), rnd(B, N, T, H, seed=64), rnd(B, N, T, H, seed=65)
    lens = torch.tensor([3, 8], dtype=torch.int32)
    binm = (torch.arange(T).view(1, T) < lens.view(B, 1)).to(torch.int32).view(B, 1, 1, T)
    a = run(q, k, v, lens=lens, len_kind=oracle.LEN_KEYLEN_I32)
    b = run(q, k, v, keep_mask=binm.expand(B, N, S, T), keep_kind=oracle.KEEP_FILTER)
    np.testing.assert_array_equal(a, b)
    # every key filtered: the filter value shifts all scores equally -> unmasked softmax
    zero = torch.zeros(B, dtype=torch.int32)
    np.testing.assert_allclose(run(q, k, v, lens=zero, len_kind=oracle.LEN_KEYLEN_I32),
                               run(q, k, v), atol=1e-12)
    filt = json.load(open(GOLDEN))["mask_filter_value_default"]["value"]
    assert Problem(q=q, k=k, v=v).mask_filter_value == filt


def test_past_split_point_does_not_change_the_result():
    B, N, S, T, H = 2, 2, 3, 9, 8
    q = rnd(B, N, S, H, seed=66)
    kt, vt = rnd(B, N, T, H, seed=67), rnd(B, N, T, H, seed=68)
    whole = run(q, kt, vt, causal=oracle.CAUSAL_LOWER_RIGHT)
    for P in (1, 4, T - 1):
        got = run(q, kt[:, :, P:], vt[:, :, P:], past_k=kt[:, :, :P], past_v=vt[:, :, :P],
                  causal=oracle.CAUSAL_LOWER_RIGHT)
        np.testing.assert_array_equal(got, whole)


def test_layout_views_do_not_change_the_result():
    B, N, S, H = 2, 3, 5, 8
    q4, k4, v4 = rnd(B, N, S, H, seed=69), rnd(B, N, S, H, seed=70), rnd(B, N, S, H, seed=71)
    q3 = q4.permute(0, 2, 1, 3).contiguous().view(B, S, N * H)
    k3 = k4.permute(0, 2, 1, 3).contiguous().view(B, S, N * H)
    v3 = v4.permute(0, 2, 1, 3).contiguous().view(B, S, N * H)
    as4 = lambda t: t.view(B, S, N, H).permute(0, 2, 1, 3)
    np.testing.assert_array_equal(run(as4(q3), as4(k3), as4(v3)), run(q4, k4, v4))


def test_fully_excluded_row_is_zero_and_sink_keeps_it_zero():
    q, k, v = rnd(1, 1, 2, 4, seed=72), rnd(1, 1, 3, 4, seed=73), rnd(1, 1, 3, 4, seed=74)
    none = torch.zeros(1, 1, 2, 3, dtype=torch.uint8)
    np.testing.assert_array_equal(run(q, k, v, keep_mask=none, keep_kind=oracle.KEEP_BOOL), 0.0)
    np.testing.assert_array_equal(run(q, k, v, keep_mask=none, keep_kind=oracle.KEEP_BOOL,
                                      head_sink=torch.tensor([1.0], dtype=torch.float64)), 0.0)


def test_projection_bias_length_matches_the_contract():
    for c in json.load(open(GOLDEN))["projection_bias_length"]["cases"]:
        assert 2 * c["N"] * c["H"] + c["N"] * c["Hv"] == c["length"]


def test_mha_projection_bias_rank4_cross_attention_takes_only_the_query_segment():
    """MultiHeadAttention ("Custom operators"): for rank-4 (cross-attention) key/value only the
    query segment of the projection bias is applied, so changing the key and value segments
    leaves Y unchanged; for rank-3 (packed) key/value every segment applies, in the order
    [query | key | value]."""
    B, N, S, T, H, Hv = 2, 3, 4, 9, 8, 4
    q, k, v = rnd(B, N, S, H, seed=131), rnd(B, N, T, H, seed=132), rnd(B, N, T, Hv, seed=133)
    bias = rnd(2 * N * H + N * Hv, seed=134)
    moved = bias.clone()
    moved[N * H:] += rnd(N * H + N * Hv, seed=135)           # other key / value segments
    seg4 = oracle.mha_projection_bias(bias, N, H, Hv, kv_rank=4)
    assert seg4[1] is None and seg4[2] is None
    y4 = run(q, k, v, q_bias=seg4[0])
    np.testing.assert_array_equal(y4, run(q, k, v, q_bias=oracle.mha_projection_bias(moved, N, H, Hv, 4)[0]))
    # the query segment does matter, and it is the first N*H values
    np.testing.assert_allclose(y4, sdpa(q + bias[:N * H].view(1, N, 1, H), k, v), atol=1e-12)
    # rank-3 key/value: all three segments, and moving the key / value segments changes Y
    qb, kb, vb = oracle.mha_projection_bias(bias, N, H, Hv, kv_rank=3)
    y3 = run(q, k, v, q_bias=qb, k_bias=kb, v_bias=vb)
    want = sdpa(q + bias[:N * H].view(1, N, 1, H), k + bias[N * H:2 * N * H].view(1, N, 1, H),
                v + bias[2 * N * H:].view(1, N, 1, Hv))
    np.testing.assert_allclose(y3, want, atol=1e-12)
    qm, km, vm = oracle.mha_projection_bias(moved, N, H, Hv, kv_rank=3)
    assert np.abs(run(q, k, v, q_bias=qm, k_bias=km, v_bias=vm) - y3).max() > 1e-3
    with pytest.raises(ValueError):
        oracle.mha_projection_bias(bias[:-1], N, H, Hv, 3)


def test_oracle_rejects_window_without_causal_and_bad_groups():
    q, k, v = rnd(1, 3, 2, 4, seed=75), rnd(1, 2, 2, 4, seed=76), rnd(1, 2, 2, 4, seed=77)
    with pytest.raises(ValueError):
        run(q, k, v)                                  # 3 query heads over 2 kv heads
    q2 = rnd(1, 2, 2, 4, seed=78)
    with pytest.raises(ValueError):
        run(q2, k, v, window=2)


# ---------------------------------------------------------------- rotary embedding (class RotaryEmbedding)

def _rope_caches(max_pos, half, base=10000.0, dtype=torch.float64):
    """cos/sin tables of RoFormer's angles pos * base^(-2d/R) (test input, not the oracle)."""
    pos = torch.arange(max_pos, dtype=torch.float64).view(-1, 1)
    inv = base ** (-torch.arange(half, dtype=torch.float64) * 2.0 / (2 * half))
    ang = pos * inv.view(1, -1)
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


def test_rotary_identity_and_quarter_turn():
    B, N, S, D = 2, 3, 4, 8
    x = rnd(B, N, S, D, seed=80)
    one, zero = torch.ones(5, D // 2, dtype=torch.float64), torch.zeros(5, D // 2, dtype=torch.float64)
    pid = torch.tensor([[0, 1, 2, 3], [4, 3, 2, 1]], dtype=torch.int64)
    for inter in (False, True):
        np.testing.assert_array_equal(oracle.rotary(x, one, zero, pid, interleaved=inter), x.numpy())
        got = oracle.rotary(x, zero, one, pid, interleaved=inter)       # 90 degrees
        xn = x.numpy()
        if inter:
            x1, x2, g1, g2 = xn[..., 0::2], xn[..., 1::2], got[..., 0::2], got[..., 1::2]
        else:
            x1, x2, g1, g2 = xn[..., :D // 2], xn[..., D // 2:], got[..., :D // 2], got[..., D // 2:]
        np.testing.assert_array_equal(g1, -x2)
        np.testing.assert_array_equal(g2, x1)


def test_rotary_equals_complex_multiplication():
    B, N, S, D = 1, 2, 6, 16
    x = rnd(B, N, S, D, seed=81)
    cos, sin = _rope_caches(32, D // 2)
    pid = torch.tensor([[5, 0, 31, 7, 7, 12]], dtype=torch.int64)
    got = oracle.rotary(x, cos, sin, pid)
    xn = x.numpy()
    z = (xn[..., :D // 2] + 1j * xn[..., D // 2:]) * np.exp(1j * np.angle(cos.numpy() + 1j * sin.numpy()))[pid.numpy()[0]]
    np.testing.assert_allclose(got[..., :D // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(got[..., D // 2:], z.imag, atol=1e-12)


def test_rotary_scores_depend_only_on_relative_position():
    D = 32
    q, k = rnd(1, 1, 1, D, seed=82), rnd(1, 1, 1, D, seed=83)
    cos, sin = _rope_caches(64, D // 2)
    def score(pq, pk):
        rq = oracle.rotary(q, cos, sin, torch.tensor([[pq]]))
        rk = oracle.rotary(k, cos, sin, torch.tensor([[pk]]))
        return float((rq * rk).sum())
    base = score(9, 4)
    for shift in (1, 7, 40):
        assert score(9 + shift, 4 + shift) == pytest.approx(base, abs=1e-10)
    assert abs(score(9, 4) - score(9, 5)) > 1e-6


def test_rotary_interleaved_is_a_channel_permutation_of_the_half_layout():
    B, N, S, D = 2, 2, 3, 12
    x = rnd(B, N, S, D, seed=84)
    cos, sin = _rope_caches(8, D // 2)
    pid = torch.tensor([[1, 2, 3], [7, 0, 5]], dtype=torch.int64)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])    # interleaved -> halves
    inter = oracle.rotary(x, cos, sin, pid, interleaved=True)
    half = oracle.rotary(x[..., perm].contiguous(), cos, sin, pid)
    np.testing.assert_allclose(inter[..., perm], half, atol=1e-14)


def test_rotary_partial_dim_passes_the_rest_and_caches_forms_agree():
    B, N, S, D, R = 2, 2, 4, 16, 8
    x = rnd(B, N, S, D, seed=85)
    cos, sin = _rope_caches(10, R // 2)
    pid = torch.tensor([[0, 3, 9, 2], [1, 1, 4, 8]], dtype=torch.int64)
    got = oracle.rotary(x, cos, sin, pid, rotary_dim=R)
    np.testing.assert_array_equal(got[..., R:], x.numpy()[..., R:])
    sub = oracle.rotary(x[..., :R].contiguous(), cos, sin, pid)
    np.testing.assert_allclose(got[..., :R], sub, atol=1e-14)
    # rank-3 caches (B, S, R/2) used directly equal rank-2 caches gathered by position ids
    cos3, sin3 = cos[pid], sin[pid]
    np.testing.assert_array_equal(oracle.rotary(x, cos3, sin3, None, rotary_dim=R), got)
    # every rotated pair keeps its length
    n_in = x.numpy()[..., :R // 2] ** 2 + x.numpy()[..., R // 2:R] ** 2
    n_out = got[..., :R // 2] ** 2 + got[..., R // 2:R] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_gqa_rotary_positions():
    """Absolute positions: a prompt without past starts at 0, a decode step after P past
    rows sits at P, seqlens_k moves the end of the valid sequence, and the query and new
    key rows end together at Tv - 1."""
    qp, kp = oracle.gqa_rotary_positions(1, 4, 4, 4)
    assert qp.tolist() == [[0, 1, 2, 3]] and kp.tolist() == [[0, 1, 2, 3]]
    qp, kp = oracle.gqa_rotary_positions(2, 1, 1, 11)
    assert qp.tolist() == [[10], [10]] and kp.tolist() == [[10], [10]]
    qp, kp = oracle.gqa_rotary_positions(2, 1, 1, 11, torch.tensor([5, 9], dtype=torch.int32))
    assert qp.tolist() == [[5], [9]] and kp.tolist() == [[5], [9]]
    qp, kp = oracle.gqa_rotary_positions(1, 3, 4, 10)
    assert qp.tolist() == [[7, 8, 9]] and kp.tolist() == [[6, 7, 8, 9]]


# ---------------------------------------------------------------- qk output (class Attention, qk_matmul_output_mode)

def _qk_case(seed=60, **kw):
    B, Nq, Nkv, S, T, H = 2, 4, 2, 6, 9, 8
    q, k, v = rnd(B, Nq, S, H, seed=seed), rnd(B, Nkv, T, H, seed=seed + 1), rnd(B, Nkv, T, H, seed=seed + 2)
    return q, k, v


def _qk_expand(k, Nq):
    return k.repeat_interleave(Nq // k.shape[1], dim=1)


def test_qk_mode0_is_the_scaled_product_whatever_the_masks():
    q, k, v = _qk_case()
    mask = rnd(2, 1, 6, 7, seed=63)                        # shorter than T: padded
    got = oracle.qk(Problem(q=q, k=k, v=v, scale=0.3, softcap=2.0, causal=oracle.CAUSAL_UPPER_LEFT,
                            add_mask=mask.expand(2, 4, 6, 7)), 0)
    want = 0.3 * torch.matmul(q, _qk_expand(k, 4).transpose(-1, -2))
    np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=1e-12)


def test_qk_mode1_adds_the_bias_and_excludes_with_minus_inf():
    q, k, v = _qk_case(seed=64)
    mask = rnd(2, 1, 6, 7, seed=67)
    pr = Problem(q=q, k=k, v=v, scale=0.3, causal=oracle.CAUSAL_UPPER_LEFT, add_mask=mask.expand(2, 4, 6, 7))
    raw = 0.3 * torch.matmul(q, _qk_expand(k, 4).transpose(-1, -2))
    want = raw.clone()
    want[..., :7] += mask
    want[..., 7:] = -math.inf                             # the padding of a short mask
    want = want.masked_fill(torch.ones(6, 9).triu(1).bool(), -math.inf)   # j > i
    np.testing.assert_array_equal(np.isinf(oracle.qk(pr, 1)), np.isinf(want.numpy()))
    np.testing.assert_allclose(oracle.qk(pr, 1), want.numpy(), rtol=0, atol=1e-12)


def test_qk_mode2_is_softcap_of_mode1_and_mode3_is_its_softmax():
    q, k, v = _qk_case(seed=68)
    pr = Problem(q=q, k=k, v=v, scale=1.7, softcap=1.5, causal=oracle.CAUSAL_LOWER_RIGHT)
    m1, m2, m3 = oracle.qk(pr, 1), oracle.qk(pr, 2), oracle.qk(pr, 3)
    fin = np.isfinite(m1)
    np.testing.assert_array_equal(fin, np.isfinite(m2))
    np.testing.assert_allclose(m2[fin], 1.5 * np.tanh(m1[fin] / 1.5), rtol=0, atol=1e-12)
    want3 = torch.softmax(torch.from_numpy(m2), dim=-1).numpy()
    np.testing.assert_allclose(m3, want3, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m3.sum(-1), 1.0, atol=1e-12)


def test_qk_probabilities_times_values_give_the_output():
    """Y = P V: the mode-3 output is the matrix the attention output averages V with,
    here with past rows, GQA, an additive mask, a window and a sink."""
    B, Nq, Nkv, S, L, P, H = 2, 4, 2, 5, 5, 4, 8
    q = rnd(B, Nq, S, H, seed=70)
    k, v = rnd(B, Nkv, L, H, seed=71), rnd(B, Nkv, L, H, seed=72)
    pk, pv = rnd(B, Nkv, P, H, seed=73), rnd(B, Nkv, P, H, seed=74)
    sink = rnd(Nq, seed=75)
    mask = rnd(B, Nq, S, P + L, seed=76)
    pr = Problem(q=q, k=k, v=v, past_k=pk, past_v=pv, causal=oracle.CAUSAL_LOWER_RIGHT, window=3,
                 head_sink=sink, add_mask=mask)
    probs = oracle.qk(pr, 3)
    vt = _qk_expand(torch.cat([pv, v], 2), Nq).numpy()
    np.testing.assert_allclose(np.einsum("bhst,bhtd->bhsd", probs, vt), oracle.attention(pr), atol=1e-12)
    # the sink takes the rest of the mass: sum_j p_j + e^sink / (sum_j e^s_j + e^sink) = 1
    logits = oracle.qk(pr, 2)
    e = np.exp(logits)                                     # exp(-inf) = 0 for excluded keys
    es = np.exp(sink.numpy())[None, :, None]
    np.testing.assert_allclose(probs.sum(-1) + es / (e.sum(-1) + es), 1.0, atol=1e-12)
    assert (probs.sum(-1) < 1.0).all()


def test_qk_fully_excluded_row_and_filter_values():
    q, k, v = _qk_case(seed=80)
    keep = torch.ones(2, 4, 6, 9, dtype=torch.uint8)
    keep[0, 1, 2] = 0                                     # one row with nothing admitted
    pr = Problem(q=q, k=k, v=v, keep_mask=keep, keep_kind=oracle.KEEP_BOOL)
    np.testing.assert_array_equal(oracle.qk(pr, 1)[0, 1, 2], -np.inf)
    np.testing.assert_array_equal(oracle.qk(pr, 3)[0, 1, 2], 0.0)
    # MultiHeadAttention key padding adds mask_filter_value instead of excluding
    lens = torch.tensor([4, 9], dtype=torch.int32)
    pr = Problem(q=q, k=k, v=v, len_kind=oracle.LEN_KEYLEN_I32, lens=lens, mask_filter_value=-50.0)
    raw, m1 = oracle.qk(pr, 0), oracle.qk(pr, 1)
    np.testing.assert_allclose(m1[0, :, :, 4:], raw[0, :, :, 4:] - 50.0, atol=1e-12)
    np.testing.assert_array_equal(m1[0, :, :, :4], raw[0, :, :, :4])
    np.testing.assert_array_equal(m1[1], raw[1])


# ---------------------------------------------------------------- backward (GroupQueryAttention gradient graph)

def _torch_grads(q, k, v, dy, **kw):
    q, k, v = (t.clone().double().requires_grad_(True) for t in (q, k, v))
    y = F.scaled_dot_product_attention(q, k, v, **kw)
    y.backward(dy.double())
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("kind", ["plain", "gqa", "causal", "float_mask", "bool_mask", "scale"])
def test_backward_equals_torch_autograd(kind):
    B, Nq, Nkv, S, T, H, Hv = 2, 4, 4, 5, 7, 8, 6
    if kind == "gqa":
        Nkv = 2
    q, k, v = rnd(B, Nq, S, H, seed=101), rnd(B, Nkv, T, H, seed=102), rnd(B, Nkv, T, Hv, seed=103)
    dy = rnd(B, Nq, S, Hv, seed=104)
    kw, tkw = {}, {}
    if kind == "gqa":
        tkw["enable_gqa"] = True
    if kind == "causal":
        kw["causal"], tkw["is_causal"] = oracle.CAUSAL_UPPER_LEFT, True
    if kind == "float_mask":
        m = rnd(B, Nq, S, T, seed=105)
        kw["add_mask"], tkw["attn_mask"] = m, m
    if kind == "bool_mask":
        keep = (rnd(B, 1, S, T, seed=106) > -0.5)
        keep[..., 0] = True                                   # every row keeps a key
        kw["keep_mask"], kw["keep_kind"] = keep.to(torch.uint8).expand(B, Nq, S, T), oracle.KEEP_BOOL
        tkw["attn_mask"] = keep
    if kind == "scale":
        kw["scale"], tkw["scale"] = 0.41, 0.41
    dq, dk, dv = oracle.backward(Problem(q=q, k=k, v=v, **kw), dy)
    wq, wk, wv = _torch_grads(q, k, v, dy, **tkw)
    for got, want in ((dq, wq), (dk, wk), (dv, wv)):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_backward_with_window_sink_and_lower_right_past_equals_autograd_of_the_definition():
    """A torch float64 forward written from the definition (the sink as an extra logit
    column with no value), differentiated by autograd."""
    B, Nq, Nkv, S, L, P, H = 1, 4, 2, 4, 4, 3, 8
    q = rnd(B, Nq, S, H, seed=110)
    k, v = rnd(B, Nkv, L, H, seed=111), rnd(B, Nkv, L, H, seed=112)
    pk, pv = rnd(B, Nkv, P, H, seed=113), rnd(B, Nkv, P, H, seed=114)
    sink, dy = rnd(Nq, seed=115), rnd(B, Nq, S, H, seed=116)
    dq, dk, dv = oracle.backward(Problem(q=q, k=k, v=v, past_k=pk, past_v=pv, causal=oracle.CAUSAL_LOWER_RIGHT,
                                         window=3, head_sink=sink), dy)
    qt = q.clone().requires_grad_(True)
    kt = torch.cat([pk, k], 2).clone().requires_grad_(True)
    vt = torch.cat([pv, v], 2).clone().requires_grad_(True)
    T = P + L
    ke, ve = kt.repeat_interleave(Nq // Nkv, 1), vt.repeat_interleave(Nq // Nkv, 1)
    s = torch.matmul(qt, ke.transpose(-1, -2)) / math.sqrt(H)
    pos = (T - S + torch.arange(S)).view(S, 1)
    j = torch.arange(T).view(1, T)
    s = s.masked_fill((j > pos) | (j < pos - 3 + 1), -math.inf)
    logits = torch.cat([s, sink.view(1, Nq, 1, 1).expand(B, Nq, S, 1)], -1)
    prob = torch.softmax(logits, -1)[..., :T]
    (torch.matmul(prob, ve) * dy).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def test_backward_with_projection_biases_equals_autograd_of_the_biased_rows():
    """MultiHeadAttention's projection-bias segments shift Q and the new K / V rows (never
    the past rows); the gradients with respect to the rows the scores see are those of
    torch's attention on the shifted rows, past rows first."""
    B, N, S, L, P, H = 2, 3, 5, 4, 3, 8
    q, k, v = rnd(B, N, S, H, seed=140), rnd(B, N, L, H, seed=141), rnd(B, N, L, H, seed=142)
    pk, pv = rnd(B, N, P, H, seed=143), rnd(B, N, P, H, seed=144)
    bq, bk, bv = rnd(N * H, seed=145), rnd(N * H, seed=146), rnd(N * H, seed=147)
    dy = rnd(B, N, S, H, seed=148)
    dq, dk, dv = oracle.backward(Problem(q=q, k=k, v=v, past_k=pk, past_v=pv, q_bias=bq, k_bias=bk, v_bias=bv,
                                         causal=oracle.CAUSAL_LOWER_RIGHT), dy)
    qs = q + bq.view(1, N, 1, H)
    ks = torch.cat([pk, k + bk.view(1, N, 1, H)], 2)
    vs = torch.cat([pv, v + bv.view(1, N, 1, H)], 2)
    T = P + L
    keep = torch.arange(T).view(1, T) <= (T - S + torch.arange(S)).view(S, 1)
    wq, wk, wv = _torch_grads(qs, ks, vs, dy, attn_mask=keep)
    assert dk.shape == (B, N, T, H) and dv.shape == (B, N, T, H)
    for got, want in ((dq, wq), (dk, wk), (dv, wv)):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_backward_matches_central_differences_of_the_forward():
    """d(sum dY * Y)/dx from the oracle backward against central differences of the oracle
    forward, with GQA, an additive mask, key lengths (filter), a boolean mask and a sink."""
    B, Nq, Nkv, S, L, H = 1, 2, 1, 3, 5, 4
    q, k, v = rnd(B, Nq, S, H, seed=120), rnd(B, Nkv, L, H, seed=121), rnd(B, Nkv, L, H, seed=122)
    mask, sink, dy = rnd(B, Nq, S, L, seed=123), rnd(Nq, seed=124), rnd(B, Nq, S, H, seed=125)
    keep = torch.ones(B, Nq, S, L, dtype=torch.uint8)
    keep[0, 1, 2, 1] = 0
    kw = dict(add_mask=mask, head_sink=sink, keep_mask=keep, keep_kind=oracle.KEEP_BOOL,
              len_kind=oracle.LEN_KEYLEN_I32, lens=torch.tensor([4], dtype=torch.int32), mask_filter_value=-3.0)
    dq, dk, dv = oracle.backward(Problem(q=q, k=k, v=v, **kw), dy)

    def loss(q_, k_, v_):
        return float((oracle.attention(Problem(q=q_, k=k_, v=v_, **kw)) * dy.numpy()).sum())

    h = 1e-6
    for name, t, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, 0, 1, 2), (0, t.shape[1] - 1, t.shape[2] - 1, t.shape[3] - 1), (0, 0, 2, 3)]:
            tp, tm = t.clone(), t.clone()
            tp[idx] += h
            tm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            assert abs(fd - g[idx]) < 1e-7, (name, idx, fd, g[idx])


def test_backward_of_rows_with_nothing_admitted_is_zero_and_softcap_is_rejected():
    q, k, v = rnd(1, 2, 4, 8, seed=130), rnd(1, 2, 6, 8, seed=131), rnd(1, 2, 6, 8, seed=132)
    dy = rnd(1, 2, 4, 8, seed=133)
    keep = torch.ones(1, 2, 4, 6, dtype=torch.uint8)
    keep[0, 0, 1] = 0
    dq, dk, dv = oracle.backward(Problem(q=q, k=k, v=v, keep_mask=keep, keep_kind=oracle.KEEP_BOOL), dy)
    np.testing.assert_array_equal(dq[0, 0, 1], 0.0)
    with pytest.raises(ValueError):
        oracle.backward(Problem(q=q, k=k, v=v, softcap=5.0), dy)
