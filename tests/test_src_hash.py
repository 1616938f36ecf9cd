"""The kernel-source hash that ties committed ncu traffic figures to the
sources they were taken on (bench.py): it ignores comments and white space,
follows every code change, and the committed decode summary's traffic line
is well formed."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def strip(text):
    return " ".join(bench._TOKENS.sub(lambda m: " " if m.group(0).startswith("/") else m.group(0),
                                      text).split())


def test_comments_and_space_do_not_count():
    a = 'int f(int x) {\n  return x / 2;  // half\n}\n'
    b = '/* doc */ int f(int x) { return x / 2; }'
    assert strip(a) == strip(b)


def test_code_and_literals_count():
    assert strip('int x = 1;') != strip('int x = 2;')
    assert strip('const char* s = "a // b";') != strip('const char* s = "a";')
    assert strip("char c = '/';") != strip("char c = '*';")


def test_committed_decode_summary_line_parses():
    """The decode summary carries a traffic line with its workload, kernel,
    bytes and source hash; the bench uses it only while the hash matches."""
    path = os.path.join(ROOT, "profiles", "decode_v1_ragged_b16_32x8_d128.md")
    lines = [x for x in open(path) if x.startswith("bench-traffic:")]
    assert len(lines) == 1
    kv = dict(x.split("=", 1) for x in lines[0].split()[1:])
    assert kv["workload"] == "ragged_b16_32x8_d128" and kv["kernel"] == "decode_partial"
    assert int(kv["bytes"]) > 110_000_000 and len(kv["src"]) == 12
    got = bench.read_traffic("ragged_b16_32x8_d128", "decode_partial")
    assert got is None or got == int(kv["bytes"]) * float(kv.get("scale", "1"))
