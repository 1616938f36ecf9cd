"""The C-ABI boundary on the host: the library builds, loads, exports every
entry point declared in include/*.h, and rejects malformed arguments before
touching the device (crucible results: malformed metadata is rejected
before device access).  No test here needs a GPU."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

from paged_kv_gqa_02_gb300 import build, ops, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        names |= set(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("pa_decode", "pa_prefill_chunk", "pa_combine"):
        assert n in names
    assert set(names) <= set(ops.EXPORTS) | {n for n in names if n.startswith("pa_")}


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert lib.pa_version() >= 100
    assert lib.pa_build_flags() == 0  # the release build: no range checks compiled in


def test_make_params_sets_every_field(lib):
    """ops.make_params accepts and stores each optional pa_params field."""
    kw = dict(deterministic=0, num_splits=3, strides=(4096, 1024, 128), decode_phases=1,
              decode_q_rows=2, sliding_window=64, decode_form=2, debug_timeout=1)
    p = ops.make_params(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=32,
                        num_pages=10, max_blocks_per_seq=4, max_context_len=128, **kw)
    assert (p.page_stride, p.token_stride, p.head_stride) == kw.pop("strides")
    for k, v in kw.items():
        assert getattr(p, k) == v, k


def test_params_struct_layout_matches_header(lib):
    """pa_params_init writes the defaults the header documents."""
    p = ops.Params()
    lib.pa_params_init(ctypes.byref(p))
    assert (p.out_dtype, p.deterministic, p.num_splits, p.page_stride) == (ops.PA_F32, 1, 0, 0)
    assert ctypes.sizeof(ops.Params) == header_layout()["sizeof"]


def header_layout():
    """sizeof(pa_params) and every field's offset, from a C compile of the header."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f for f, _ in ops.Params._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"paged_gqa.h\"\nint main(void) {\n"
    src += 'printf("sizeof %zu\\n", sizeof(pa_params));\n'
    src += "".join(f'printf("{n} %zu\\n", offsetof(pa_params, {n}));\n' for n in names)
    src += "return 0; }\n"
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(c, "w") as f:
            f.write(src)
        subprocess.run([cc, "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


def test_params_field_offsets_match_header():
    """The ctypes binding's pa_params has the header's field offsets."""
    layout = header_layout()
    for name, _ in ops.Params._fields_:
        assert getattr(ops.Params, name).offset == layout[name], name


def test_status_strings(lib):
    for code, name in ops.STATUS.items():
        assert lib.pa_status_string(code).decode().startswith(name)


def base_params(**kw):
    args = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=32,
                num_pages=64, max_blocks_per_seq=16, max_context_len=512, dtype="bf16")
    args.update(kw)
    return ops.make_params(**args)


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first


def call_decode(p, q=FAKE, out=FAKE, bt=FAKE, ws=None, nbytes=0):
    return ops.load().pa_decode(ctypes.byref(p), q, FAKE, FAKE, bt, FAKE, out, ws, nbytes, None, None)


@pytest.mark.parametrize("field,value,code", [
    ("num_seqs", 0, 2), ("num_q_heads", 7, 2), ("num_kv_heads", 0, 2),
    ("head_dim", 96, 6), ("page_size", 8, 6), ("num_q_heads", 2 * 17, 6),
    ("max_context_len", 16 * 32 + 1, 2), ("num_pages", 0, 2), ("q_dtype", 9, 3),
    ("kv_dtype", ops.PA_F16, 6), ("out_dtype", ops.PA_BF16, 6), ("deterministic", 2, 2),
    ("num_splits", -1, 2), ("head_stride", 4, 4), ("token_stride", 100, 4),
    ("decode_phases", 4, 2), ("decode_phases", -1, 2), ("decode_form", 3, 2),
    ("decode_form", -1, 2), ("debug_timeout", 2, 2),
])
def test_rejects_bad_params(lib, field, value, code):
    p = base_params()
    if field == "num_q_heads" and value == 34:
        p.num_kv_heads = 2
    setattr(p, field, value)
    assert call_decode(p) == code


def test_rejects_null_and_misaligned(lib):
    p = base_params()
    assert call_decode(p, q=None) == 1
    assert call_decode(p, out=ctypes.c_void_p((1 << 20) + 4)) == 4
    assert call_decode(p, bt=ctypes.c_void_p((1 << 20) + 2)) == 4


def test_combine_host_checks(lib):
    """pa_combine rejects NULL pointers, a split stride below 1, head_dim 256
    and misaligned partials, out or split counts before launching."""
    p = base_params()
    L = ops.load()
    big = ctypes.c_void_p(1 << 20)

    def call(ml=big, acc=big, S=4, spl=None, out=big):
        return L.pa_combine(ctypes.byref(p), ml, acc, S, spl, out, None)
    assert call(ml=None) == 1 and call(acc=None) == 1 and call(out=None) == 1
    assert call(S=0) == 2
    assert call(acc=ctypes.c_void_p((1 << 20) + 8)) == 4
    assert call(out=ctypes.c_void_p((1 << 20) + 4)) == 4
    assert call(ml=ctypes.c_void_p((1 << 20) + 4)) == 4
    assert call(spl=ctypes.c_void_p((1 << 20) + 2)) == 4
    p.head_dim = 256
    assert call() == 6


def test_rejects_small_workspace(lib):
    p = base_params(max_context_len=512)
    S, tok = ops.decode_plan(p)
    assert S > 1
    need = ops.decode_workspace_size(p)
    assert need >= 2 * 8 * S * (128 + 2) * 4
    assert call_decode(p, ws=FAKE, nbytes=need - 1) == 5
    assert call_decode(p, ws=None, nbytes=0) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(decode_q_rows=17), 2),                                  # more rows than supported
    (dict(decode_q_rows=-1), 2),
    (dict(decode_q_rows=9, max_context_len=8), 2),                # rows beyond the capacity
    (dict(sliding_window=-1), 2),
    (dict(dtype="f32", sliding_window=8), 6),                     # windows: split-KV kernel only
    (dict(num_splits=2, sliding_window=8), 6),
    (dict(head_dim=256, num_q_heads=32, num_kv_heads=2), 6),      # D 256 with 16 heads a kv head
    (dict(head_dim=256, num_splits=2), 6),                        # D 256 off the split-KV kernel
])
def test_rejects_unsupported_decode_options(lib, kw, code):
    assert call_decode(base_params(**kw)) == code


def test_partial_and_append_reject_several_rows(lib):
    p = base_params(decode_q_rows=2)
    S, _ = ops.decode_plan(p)
    assert lib.pa_decode_partial(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, S,
                                 None, None) == 6
    assert ops.load().pa_decode_append(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                       None, 0, None, None) == 6


def test_row_block_workspace_holds_every_block(lib):
    """16-bit K/V, 8 q heads a kv head, 4 rows: two row blocks of 2 rows are
    units of one launch, each with 16 columns, so the workspace holds a slot
    per (part, unit) for 2 x num_kv_heads units a sequence."""
    p = base_params(num_q_heads=32, num_kv_heads=4, decode_q_rows=4)
    need = ops.decode_workspace_size(p)
    slots = 152 * 8 + 2 * 4 * 2
    assert need >= slots * 16 * (128 + 2) * 4
    assert need > ops.decode_workspace_size(base_params(num_q_heads=32, num_kv_heads=4))
    assert call_decode(p, ws=FAKE, nbytes=need - 1) == 5


def test_fp32_multi_row_workspace_holds_every_row(lib):
    """fp32 K/V with several query rows: split partials per (row, q head), so
    the workspace grows with the rows and a smaller one is refused."""
    p1 = base_params(dtype="f32")
    p3 = base_params(dtype="f32", decode_q_rows=3)
    S, _ = ops.decode_plan(p3)
    assert S > 1 and ops.decode_plan(p1)[0] == S
    need = ops.decode_workspace_size(p3)
    assert need >= 2 * 3 * 8 * S * (128 + 2) * 4
    assert need > ops.decode_workspace_size(p1)
    assert call_decode(p3, ws=FAKE, nbytes=need - 1) == 5
    assert call_decode(p3, ws=None, nbytes=0) == 1


def test_partial_rejects_wrong_split_count(lib):
    p = base_params()
    S, _ = ops.decode_plan(p)
    rc = lib.pa_decode_partial(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, S + 1,
                               None, None)
    assert rc == 2


def test_prefill_rejects_bad_sizes(lib):
    p = base_params()
    L = lib
    assert L.pa_prefill_chunk(ctypes.byref(p), FAKE, None, 4, 4, FAKE, FAKE, FAKE, FAKE, FAKE,
                              None, 0, None, None) == 1
    assert L.pa_prefill_chunk(ctypes.byref(p), FAKE, FAKE, 0, 4, FAKE, FAKE, FAKE, FAKE, FAKE,
                              None, 0, None, None) == 2
    assert L.pa_prefill_chunk(ctypes.byref(p), FAKE, FAKE, 4, 513, FAKE, FAKE, FAKE, FAKE, FAKE,
                              None, 0, None, None) == 2


def test_split_plan_is_a_function_of_params(lib):
    """Deterministic plans: whole pages per split, enough splits to cover the
    capacity, same answer every call (the grid never depends on device data;
    crucible README: split count fixed at capacity for graph replay)."""
    for wl in workloads.ALL[:4]:
        p = ops.params_for(wl)
        S, tok = ops.decode_plan(p)
        assert tok % wl.page_size == 0 and S * tok >= p.max_context_len > (S - 1) * tok
        assert ops.decode_plan(p) == (S, tok)
        p2 = ops.params_for(wl, num_splits=3)
        S2, tok2 = ops.decode_plan(p2)
        assert S2 <= 3 and S2 * tok2 >= p2.max_context_len
