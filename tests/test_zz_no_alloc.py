"""The allocation-free decode entry point, sdpa_attn_decode_static.

It serves callers that cannot allocate device memory themselves (a host framework that
owns the whole device memory budget and gives its plugins no allocator, or a serving loop
that cannot pay for cudaMalloc's device-wide synchronisation): instead of a caller
workspace it keeps the decode partials in a fixed device array inside the library.
These tests check, through the C ABI, that on consecutive calls (the array keeps the
previous call's contents) its results are bit-identical to sdpa_attn_decode with a
workspace (the same kernels on the same partials) and match the oracle, also on a problem
whose partials fill most of the array; and that problems whose partials do not fit are
rejected before any launch.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from scaled_dot_product_gb300 import sdpa
from scaled_dot_product_gb300.workloads import as4d, make_case, workload

TOL = {torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}


def _decode_cases():
    a = workload(4, small=True)                                 # MHA fp16, key lengths, present
    b = make_case("gqa_decode", dtype=torch.bfloat16, B=3, Nq=8, Nkv=2, S=2, L=2, P=333, H=64,
                  seed=77, causal="lower_right", window=100, sink=True, want_present=True,
                  q_layout="bsnh")
    # partials of 7.6 MiB: the top of the 8 MiB array is in use
    c = make_case("gqa_decode_near_scratch_limit", dtype=torch.float16, B=2, Nq=64, Nkv=4, S=8, L=8,
                  P=14990, H=128, seed=78, causal="lower_right", want_present=True)
    return [a, b, c]


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def _with_workspace(dcase):
    y, pk, pv = sdpa.run_case(dcase, "decode", workspace=sdpa.case_workspace(dcase, "decode"))
    return y.clone(), pk.clone(), pv.clone()


def _static(dcase):
    y_store, y4, pk, pv = sdpa.case_outputs(dcase)
    q, k, v = dcase.views()
    sdpa.sdpa_attn_decode_static(q, k, v, y=y4, **sdpa.case_kwargs(dcase, pk, pv))
    return y_store, pk, pv


@pytest.mark.gpu
def test_static_decode_matches_workspace_decode_and_oracle_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from oracle_adapter import expected_present, problem
    from scaled_dot_product_gb300 import build
    build.build()
    host = _decode_cases()
    cases = [c.to("cuda") for c in host]
    assert sdpa.sdpa_workspace_size(sdpa.make_params(*cases[2].views(), y=sdpa.case_outputs(cases[2])[1],
                                                     **sdpa.case_kwargs(cases[2]))[0],
                                     sdpa.SDPA_OP_DECODE) > (7 << 20)
    refs = [_with_workspace(c) for c in cases]
    want = [oracle.attention(problem(c)) for c in host]
    present = [expected_present(c) for c in host]
    # calls in a row on different problems, then the first ones again: every call finds the
    # previous call's partials in the shared array
    for n, i in enumerate([0, 1, 2, 0, 2, 1]):
        y, pk, pv = _static(cases[i])
        torch.cuda.synchronize()
        assert sdpa.sdpa_query_status() == sdpa.SDPA_OK
        ry, rk, rv = refs[i]
        assert torch.equal(_bits(y), _bits(ry)), f"call {n}: differs from the workspace decode"
        got = as4d(y.float().cpu(), host[i].q_layout, host[i].Nq).double().numpy()
        err = np.abs(got - want[i]).max()
        assert err <= TOL[host[i].dtype], f"call {n}: max-abs error {err:.3e} against the oracle"
        ek, ev = present[i]
        assert torch.equal(_bits(pk.cpu()), _bits(ek)) and torch.equal(_bits(pv.cpu()), _bits(ev))
        assert torch.equal(_bits(pk), _bits(rk)) and torch.equal(_bits(pv), _bits(rv))


def test_static_decode_rejects_partials_beyond_the_scratch():
    sdpa_build = pytest.importorskip("scaled_dot_product_gb300.build")
    sdpa_build.build()
    # 32768 query rows over 4096 keys need far more than the built-in 8 MiB; the input
    # views overlap a small buffer (inputs may alias each other) so nothing large is held
    B, N, S, P, H = 64, 32, 16, 4080, 128
    store = torch.zeros(1 << 16, dtype=torch.float16)
    view = lambda s: store.as_strided((B, N, s, H), (8, 8, 8, 1))
    y = torch.zeros(B, N, S, H, dtype=torch.float16)
    params, keep = sdpa.make_params(view(S), view(S), view(S), y=y, past_k=view(P), past_v=view(P))
    assert sdpa.sdpa_workspace_size(params, sdpa.SDPA_OP_DECODE) > (8 << 20)
    rc = sdpa.lib().sdpa_attn_decode_static(ctypes.byref(params), None)
    assert rc == sdpa.SDPA_ERR_WORKSPACE
    assert "built-in scratch" in sdpa.sdpa_last_error()


def test_static_decode_binding_requires_the_output():
    # the Python binding allocates nothing either: the caller passes y
    q = torch.zeros(1, 1, 1, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="y"):
        sdpa.sdpa_attn_decode_static(q, q, q)
