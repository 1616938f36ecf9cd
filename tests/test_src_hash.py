"""The kernel-source hash that ties committed ncu traffic figures to the
sources they were taken on (bench.py): it covers the kernel's translation
unit and the local headers it includes, ignores comments and white space,
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
    assert kv["workload"] == "ragged_b16_32x8_d128" and kv["kernel"] == "decode_v1"
    assert int(kv["bytes"]) > 110_000_000 and len(kv["src"]) == 12
    got = bench.read_traffic("ragged_b16_32x8_d128", "decode_v1")
    assert got is None or got == int(kv["bytes"]) * float(kv.get("scale", "1"))


def test_kernel_sources_follow_includes():
    """Each kernel's hash covers its own file and the headers it includes,
    the public header among them, and no other kernel's file."""
    names = lambda k: {os.path.basename(f) for f in bench.kernel_sources(k)}
    dec, pre = names("decode_v1"), names("prefill_tc")
    assert {"pa_decode_v1.cu", "pa_ptx.cuh", "pa_common.cuh", "paged_gqa.h"} <= dec
    assert "pa_prefill_tc.cu" not in dec and "pa_tc.cuh" not in dec
    assert {"pa_prefill_tc.cu", "pa_tc.cuh", "pa_ptx.cuh"} <= pre and "pa_decode_v1.cu" not in pre
    assert bench.src_hash("decode_v1") != bench.src_hash("prefill_tc")
    assert bench.read_traffic("ragged_b16_32x8_d128", "no_such_kernel") is None
