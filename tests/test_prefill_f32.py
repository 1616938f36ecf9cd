"""Chunked prefill with fp32 Q/K/V (the register-tiled CUDA-core kernel)
against the fp64 oracle, through the C ABI: every group size up to 16, both
head dims and page sizes, chunks over history spanning several 64-key
blocks, row tiles the rows do not fill, and the device-error paths (pages
outside the pool, invalid lengths, NaN in memory no row may read).
Tolerance: max abs <= 1e-5 (fp32 K/V)."""
from __future__ import annotations

import os
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, ops, workloads
from helpers import problem, assert_within, bitwise_equal
from test_gpu_parity import gpu_prefill

pytestmark = pytest.mark.gpu

TOL = workloads.TOL_F32
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


CASES = [
    # B, Hq, Hkv, D, P, lens, qlens
    (1, 4, 1, 64, 16, (1,), (1,)),                       # one row, one key
    (2, 12, 3, 64, 16, (100, 300), (37, 300)),           # G 4, history + chunk, several key blocks
    (3, 16, 16, 64, 32, (64, 65, 129), (64, 1, 65)),     # G 1: 64 rows a tile
    (2, 15, 5, 128, 16, (513, 77), (130, 77)),           # G 3: 21 rows x 3 heads = 63 of 64
    (2, 40, 8, 128, 32, (1000, 31), (250, 31)),          # G 5: 12 rows a tile, ragged tails
    (2, 64, 8, 64, 32, (333, 2049), (100, 9)),           # G 8
    (1, 32, 2, 128, 16, (700,), (700,)),                 # G 16: 4 rows a tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-P{c[4]}")
def test_prefill_f32_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, qlens = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, qlens=qlens, dt="f32",
                        num_pages=sum((L + P - 1) // P for L in lens) + 3,
                        seed=zlib.crc32(repr(case).encode()) & 0xFFFF)
    got, status = gpu_prefill(inp, meta)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL, f"f32 prefill {case}")


def test_prefill_f32_run_to_run_and_permuted_pages_bitwise():
    inp, meta = problem(B=2, Hq=12, Hkv=3, D=64, P=16, lens=(400, 170), qlens=(200, 170), dt="f32",
                        num_pages=40, seed=21)
    a, _ = gpu_prefill(inp, meta)
    assert bitwise_equal(gpu_prefill(inp, meta)[0], a)
    # the same data behind another physical page order
    perm = np.random.default_rng(5).permutation(int(inp["num_pages"]))
    moved = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy(),
                 block_tables=inp["block_tables"].copy())
    moved["k_cache"][perm] = inp["k_cache"]
    moved["v_cache"][perm] = inp["v_cache"]
    bt = moved["block_tables"]
    bt[bt >= 0] = perm[bt[bt >= 0]]
    assert bitwise_equal(gpu_prefill(moved, meta)[0], a)


def test_prefill_f32_poisoned_unread_memory_changes_nothing():
    """NaN in unreferenced pages and in the slots past each context in its
    last page never reach the output."""
    P = 16
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=P, lens=(45, 200, 97), qlens=(45, 20, 60), dt="f32",
                        num_pages=24, seed=43)
    base, st0 = gpu_prefill(inp, meta)
    pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    used = set(int(x) for x in inp["block_tables"].reshape(-1) if x >= 0)
    for pg in range(int(inp["num_pages"])):
        if pg not in used:
            pois["k_cache"][pg] = np.nan
            pois["v_cache"][pg] = np.nan
    for s, L in enumerate(inp["context_lens"]):
        last = inp["block_tables"][s][(L - 1) // P]
        if L % P:
            pois["k_cache"][last, L % P:] = np.nan
            pois["v_cache"][last, L % P:] = np.nan
    got, status = gpu_prefill(pois, meta)
    assert st0 == 0 and status == 0 and bitwise_equal(got, base)
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL, "poisoned")


def test_prefill_f32_bad_page_flags_and_skips():
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=64, P=32, lens=(300, 300), qlens=(40, 40), dt="f32",
                        num_pages=20, seed=65)
    bad = dict(inp, block_tables=inp["block_tables"].copy())
    bad["block_tables"][1, 2] = 5000  # outside the pool
    got, status = gpu_prefill(bad, meta)
    assert status == ops.PA_DEV_BAD_PAGE
    assert np.isfinite(got).all()
    assert_within(got[:40], oracle.attention(inp, threads=THREADS, **meta)[:40], TOL, "unaffected sequence")


def test_prefill_f32_bad_length_flags_and_zeroes():
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=64, P=16, lens=(64, 64), qlens=(32, 32), dt="f32",
                        num_pages=10, seed=67)
    bad = dict(inp, context_lens=np.array([64, 10], dtype=np.int32))  # L < chunk rows
    got, status = gpu_prefill(bad, meta)
    assert status == ops.PA_DEV_BAD_LEN
    assert np.array_equal(got[32:], np.zeros_like(got[32:]))
    assert_within(got[:32], oracle.attention(inp, threads=THREADS, **meta)[:32], TOL, "valid sequence")
