"""Host logic of bench.py that needs no GPU: the comment-free source digest that decides
whether a committed DRAM-traffic figure still describes the kernel, and the work model
behind every reported TFLOP/s."""
import json
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle_adapter import problem

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from scaled_dot_product_gb300.workloads import make_case  # noqa: E402


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // line comment\n'
           '/* block\n   comment */ int b = 2;\n'
           'const char* s = "not // a comment /* either */";\n'
           "char c = '/';  /* trailing */\n"
           '\n'
           'asm("mov.u64 %0, %%globaltimer;" : "=l"(t));   // timer\n')
    out = bench.strip_comments(src)
    assert out.splitlines() == [
        'int a = 1;',
        '  int b = 2;',
        'const char* s = "not // a comment /* either */";',
        "char c = '/';",
        'asm("mov.u64 %0, %%globaltimer;" : "=l"(t));',
    ]


def test_digest_ignores_comment_edits_and_sees_code_edits():
    csrc = os.path.join(ROOT, "scaled_dot_product_gb300", "csrc")
    base = {n: open(os.path.join(csrc, n), encoding="utf-8").read() for n in bench.KERNEL_SOURCES["rotary"]}
    d0 = bench.source_digest("rotary", read=lambda n: base[n])
    assert d0 == bench.source_digest("rotary")
    commented = dict(base, **{"rotary.cu": "// a new remark\n" + base["rotary.cu"].replace("\n", "  /* x */\n", 1)})
    assert bench.source_digest("rotary", read=lambda n: commented[n]) == d0
    changed = dict(base, **{"rotary.cu": base["rotary.cu"] + "\nstatic int unused_marker;\n"})
    assert bench.source_digest("rotary", read=lambda n: changed[n]) != d0


def test_committed_traffic_figures_are_reported_only_for_their_sources():
    """bench reports a figure of profiles/ncu_traffic.json only while the kernel family's
    sources, without comments, hash to the digest recorded with it; after a code change the
    figure is null until it is captured again."""
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, entry in d.items():
        if name.startswith("_"):
            continue
        current = bench.source_digest(name) == entry["source_digest"]
        assert bench.ncu_traffic(name) == (entry["dram_bytes_per_launch"] if current else None), name



@pytest.mark.parametrize("kw", [
    dict(causal="upper_left"),
    dict(causal="lower_right", L=37),
    dict(causal="lower_right", window=5, L=40),
    dict(causal="upper_left", window=3, len_kind="nonpad", len_range=(1, 23)),
    dict(causal="lower_right", len_kind="seqlens_k", len_range=(10, 22), P=9),
    dict(causal="none", len_kind="nonpad", len_range=(0, 23)),
])
def test_work_model_counts_the_keys_the_oracle_admits(kw):
    """bench.admitted_pairs_per_row, the work behind every reported TFLOP/s, equals the number
    of keys per query row that the oracle's rules admit (stage 1 of the qk output: an excluded
    key is -inf)."""
    kw = dict(kw)
    L = kw.pop("L", 23)
    c = make_case("work", dtype=torch.float32, B=2, Nq=2, Nkv=1, S=19, L=L, H=8, seed=5, **kw)
    want = np.isfinite(oracle.qk(problem(c), 1)).sum(axis=-1)          # (B, Nq, S)
    got = bench.admitted_pairs_per_row(c)                              # (B, S)
    for h in range(c.Nq):
        np.testing.assert_array_equal(got, want[:, h, :])
