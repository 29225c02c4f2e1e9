"""Host logic of bench.py that needs no GPU: the comment-free source digest that decides
whether a committed DRAM-traffic figure still describes the kernel."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


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


def test_committed_traffic_figures_match_the_sources():
    """Every figure in profiles/ncu_traffic.json was taken on sources that, without
    comments, are today's: bench reports it (a code change would make it null)."""
    import json
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, entry in d.items():
        if name.startswith("_"):
            continue
        assert bench.source_digest(name) == entry["source_digest"], name
        assert bench.ncu_traffic(name) == entry["dram_bytes_per_launch"], name
