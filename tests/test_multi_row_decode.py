"""pa_decode with several query rows per sequence (decode_q_rows > 1), against
the fp64 oracle, through the C ABI.

Row t of T rows of a sequence of length L attends keys [0, L - T + t], the
chunked-prefill rule, so the oracle is the one used for prefill on the same
packed rows.  16-bit K/V run on the split-KV kernel with the rows as extra
MMA columns, in blocks of 16 / (Hq/Hkv) rows; fp32 on the CUDA-core pass
over row tiles x key splits and the combine.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, ops, workloads
from helpers import problem, assert_within, bitwise_equal

pytestmark = pytest.mark.gpu

TOL = {"f32": workloads.TOL_F32, "f16": workloads.TOL_16, "bf16": workloads.TOL_16}
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def run_rows(inp, meta, T, **kw):
    B, P = len(inp["context_lens"]), meta["page_size"]
    bt = inp["block_tables"]
    p = ops.make_params(num_seqs=B, num_q_heads=meta["num_q_heads"], num_kv_heads=meta["num_kv_heads"],
                        head_dim=meta["head_dim"], page_size=P, num_pages=int(inp["num_pages"]),
                        max_blocks_per_seq=bt.shape[1], max_context_len=bt.shape[1] * P,
                        scale=meta["scale"], dtype=meta["q_dtype"], kv_dtype=meta["kv_dtype"],
                        decode_q_rows=T, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


CASES = [
    # B, Hq, Hkv, D, P, lens, T, dtype
    (4, 16, 4, 128, 32, (2, 31, 33, 700), 2, "bf16"),     # 8 columns: one MMA column tile
    (3, 16, 4, 128, 32, (4, 100, 1500), 4, "f16"),        # 16 columns: two tiles
    (2, 32, 4, 128, 16, (33, 900), 2, "bf16"),            # G 8 x 2 rows, 16-slot pages
    (2, 28, 4, 64, 16, (17, 300), 2, "f16"),              # G 7 x 2 rows, D 64
    (3, 16, 4, 128, 32, (4, 33, 65), 4, "bf16"),          # rows whose keys end before the last page
    (2, 32, 4, 128, 32, (9, 400), 4, "bf16"),             # G 8 x 4 rows: two row blocks of 2
    (2, 40, 8, 128, 32, (5, 1000), 5, "f16"),             # G 5 x 5 rows: blocks of 3 and 2
    (2, 32, 2, 64, 16, (3, 200), 3, "bf16"),              # G 16: one row per block
    (2, 12, 3, 64, 16, (3, 100), 3, "f32"),               # fp32: the CUDA-core pass
    (3, 12, 3, 64, 16, (5, 333, 1024), 5, "f32"),         # fp32: row tiles of 4 and 1, many key splits
    (2, 32, 4, 128, 32, (16, 700), 16, "f32"),            # fp32: 16 rows, G 8
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-P{c[4]}-T{c[6]}-{c[7]}")
def test_multi_row_decode_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, T, dt = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, qlens=(T,) * B, dt=dt,
                        num_pages=sum((L + P - 1) // P for L in lens) + 7, seed=33)
    got, status = run_rows(inp, meta, T)
    assert status == 0
    ref = oracle.attention(inp, threads=THREADS, **meta)
    assert_within(got, ref, TOL[dt], f"T={T}")


def test_multi_row_decode_run_to_run_bitwise():
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=32, lens=(4, 600, 2000), qlens=(4,) * 3, dt="bf16",
                        num_pages=100, seed=34)
    a, _ = run_rows(inp, meta, 4)
    b, _ = run_rows(inp, meta, 4)
    assert bitwise_equal(a, b)


def test_multi_row_decode_short_sequence_is_flagged():
    """L < T is an invalid length: its rows are zeros and PA_DEV_BAD_LEN is set."""
    inp, meta = problem(B=2, Hq=16, Hkv=4, D=128, P=32, lens=(3, 50), qlens=(3, 3), dt="bf16",
                        num_pages=8, seed=35)
    ref = oracle.attention(inp, threads=THREADS, **meta)  # sequence 1 is the same in both
    bad = dict(inp)
    bad["context_lens"] = np.array([2, 50], dtype=np.int32)  # sequence 0: fewer keys than rows
    got, status = run_rows(bad, meta, 3)
    assert status == 2  # PA_DEV_BAD_LEN alone
    assert np.all(got[:3] == 0)
    assert_within(got[3:], ref[3:], TOL["bf16"], "valid sequence beside an invalid one")


def test_multi_row_decode_phases_split_the_call():
    """decode_phases 1 then 2 on one workspace gives the single call's result
    bit for bit, with the rows in two blocks (G 8 x 4 rows) of one launch."""
    inp, meta = problem(B=2, Hq=32, Hkv=4, D=128, P=32, lens=(9, 900), qlens=(4, 4), dt="bf16",
                        num_pages=40, seed=37)
    whole, _ = run_rows(inp, meta, 4)
    bt = inp["block_tables"]
    p = ops.make_params(num_seqs=2, num_q_heads=32, num_kv_heads=4, head_dim=128, page_size=32,
                        num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                        max_context_len=bt.shape[1] * 32, scale=meta["scale"], dtype="bf16",
                        kv_dtype="bf16", decode_q_rows=4)
    d = ops.device_inputs(inp, "bf16")
    ws = torch.zeros(ops.decode_workspace_size(p), dtype=torch.uint8, device="cuda")
    out = torch.full((8, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
    for ph in (1, 2):
        p.decode_phases = ph
        ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], out=out,
                   workspace=ws)
    torch.cuda.synchronize()
    assert bitwise_equal(out.cpu().numpy(), whole)


def test_multi_row_decode_fp32_run_to_run_bitwise():
    inp, meta = problem(B=2, Hq=12, Hkv=3, D=64, P=16, lens=(7, 1000), qlens=(4, 4), dt="f32",
                        num_pages=80, seed=36)
    a, _ = run_rows(inp, meta, 4)
    b, _ = run_rows(inp, meta, 4)
    assert bitwise_equal(a, b)


@pytest.mark.parametrize("T", [2, 4])
def test_multi_row_decode_full_size_fp32(T):
    """Crucible's decode shape (12 q / 3 kv heads, D64, context 1024, P16,
    fp32) with T query rows: key splits x row tiles, then the combine."""
    wl = workloads.BY_NAME["decode_12x3_d64_L1024"]
    inp = wl.make_inputs(q_lens=(T,) * wl.num_seqs)
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, status = run_rows(inp, meta, T)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL["f32"], f"fp32 T={T}")


def test_multi_row_decode_full_size_ragged_batch():
    """The ragged 16-sequence decode batch (32 q / 8 kv heads, D128, P32,
    bf16) with two query rows per sequence."""
    wl = workloads.BY_NAME["ragged_b16_32x8_d128"]
    T = 2
    lens = tuple(max(L, T) for L in wl.context_lens)
    inp = wl.make_inputs(q_lens=(T,) * wl.num_seqs, context_lens=lens)
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, status = run_rows(inp, meta, T)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL["bf16"], "ragged T=2")
