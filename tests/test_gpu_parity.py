"""CUDA path vs the fp64 oracle, through the C ABI (ctypes binding).

Tolerances (element by element, fp32 output):
  fp32 K/V:      max abs <= 1e-5
  f16/bf16 K/V:  max abs <= 2e-3 and max rel <= 1e-2 where |ref| > 1e-2
Bitwise checks: a permuted block table over the same data, run-to-run
repetition, and poisoned never-read memory all give identical output bits.
"""
from __future__ import annotations

import math
import os
import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, inputs, ops, workloads
from helpers import problem, assert_within, bitwise_equal

pytestmark = pytest.mark.gpu

TOL = {"f32": workloads.TOL_F32, "f16": workloads.TOL_16, "bf16": workloads.TOL_16}
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def params_of(inp, meta, **kw):
    P = meta["page_size"]
    bt = inp["block_tables"]
    args = dict(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"], page_size=P,
                num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                max_context_len=bt.shape[1] * P, scale=meta["scale"], dtype=meta["q_dtype"],
                kv_dtype=meta["kv_dtype"])
    args.update(kw)
    return ops.make_params(**args)


def gpu_decode(inp, meta, **kw):
    p = params_of(inp, meta, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


def gpu_prefill(inp, meta, **kw):
    p = params_of(inp, meta, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    qlens = np.diff(inp["cu_q_lens"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.prefill_chunk(p, d["q"], d["cu_q_lens"], int(inp["cu_q_lens"][-1]),
                            int(qlens.max()), d["k_cache"], d["v_cache"], d["block_tables"],
                            d["context_lens"], dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


# ----------------------------------------------------------- small shapes --

DECODE_CASES = [
    # B, Hq, Hkv, D, P, lens, dtype
    (1, 4, 1, 64, 16, (1,), "f32"),
    (3, 12, 3, 64, 16, (1, 17, 1024), "f32"),
    (2, 8, 8, 128, 32, (31, 33), "f16"),
    (4, 28, 4, 128, 32, (1, 32, 64, 700), "f16"),
    (3, 40, 8, 128, 32, (5, 333, 1641), "f16"),
    (5, 32, 8, 128, 32, (1, 31, 32, 33, 2000), "bf16"),
    (2, 32, 2, 128, 16, (15, 1000), "bf16"),
    (2, 14, 2, 64, 32, (63, 65), "bf16"),
    (2, 10, 2, 64, 16, (129, 257), "f16"),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-P{c[4]}-{c[6]}")
def test_decode_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, dt = case
    npages = sum((L + P - 1) // P for L in lens) + 7
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt, num_pages=npages,
                        seed=zlib.crc32(repr(case).encode()) & 0xFFFF)
    got, status = gpu_decode(inp, meta)
    assert status == 0
    ref = oracle.attention(inp, threads=THREADS, **meta)
    assert_within(got, ref, TOL[dt], f"decode {case}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_decode_split_counts(splits):
    """Every split count gives the oracle's answer (split-KV + combine)."""
    inp, meta = problem(B=3, Hq=20, Hkv=4, D=128, P=32, lens=(1, 500, 2047), dt="bf16",
                        num_pages=200, seed=77)
    got, status = gpu_decode(inp, meta, num_splits=splits)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL["bf16"], f"S={splits}")


PREFILL_CASES = [
    # B, Hq, Hkv, D, P, lens, qlens, dtype
    (1, 4, 1, 64, 16, (16,), (16,), "f32"),
    (2, 12, 3, 64, 16, (100, 37), (37, 37), "f32"),
    (3, 16, 2, 128, 32, (300, 64, 33), (9, 64, 1), "bf16"),
    (2, 64, 8, 128, 32, (160, 96), (96, 32), "bf16"),
    (4, 28, 4, 128, 32, (17, 64, 129, 257), (17, 64, 129, 257), "f16"),
    # tensor-core path: every group size, both page sizes, row tiles that
    # leave rows unused, chunks spanning several key tiles and a ragged tail
    (2, 16, 16, 128, 16, (300, 129), (300, 1), "bf16"),
    (3, 32, 16, 128, 32, (1000, 517, 64), (200, 17, 64), "f16"),
    (2, 64, 16, 128, 16, (777, 2048), (130, 33), "bf16"),
    (1, 32, 2, 128, 32, (1500,), (100,), "bf16"),
    (2, 24, 2, 128, 32, (400, 260), (260, 260), "f16"),
    (2, 40, 8, 128, 16, (129, 3000), (129, 77), "f16"),
    # tensor-core path at head_dim 64 (one 64-dim half a row): several group
    # sizes and both page sizes
    (2, 12, 3, 64, 16, (100, 300), (37, 300), "bf16"),
    (3, 32, 4, 64, 32, (1000, 64, 129), (300, 64, 1), "f16"),
    (2, 16, 16, 64, 32, (257, 2000), (257, 50), "bf16"),
    (1, 40, 8, 64, 16, (3000,), (129,), "f16"),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-{c[7]}")
def test_prefill_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, qlens, dt = case
    npages = sum((L + P - 1) // P for L in lens) + 3
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, qlens=qlens, dt=dt,
                        num_pages=npages, seed=zlib.crc32(repr(case).encode()) & 0xFFFF)
    got, status = gpu_prefill(inp, meta)
    assert status == 0
    ref = oracle.attention(inp, threads=THREADS, **meta)
    assert_within(got, ref, TOL[dt], f"prefill {case}")


# ------------------------------------------------------------ the configs --

@pytest.mark.parametrize("wl", workloads.ALL[:4], ids=lambda w: w.name)
def test_decode_workload_full(wl):
    inp = wl.make_inputs()
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, status = gpu_decode(inp, meta, max_context_len=wl.max_blocks_per_seq * wl.page_size)
    assert status == 0
    ref = oracle.attention(inp, wl, threads=THREADS)
    assert_within(got, ref, wl.tol, wl.name)


def test_prefill_workload_full():
    """The 8 x (2048 + 512) prefill at full size, compared with the oracle
    element by element: all 4,096 rows x 64 q heads x 128 dims (the oracle
    takes about 1.5e11 fp64 multiply-adds, spread over the host's cores)."""
    wl = workloads.C5
    inp = wl.make_inputs()
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, status = gpu_prefill(inp, meta)
    assert status == 0
    assert got.shape == (wl.total_q, wl.num_q_heads, wl.head_dim)
    ref = oracle.attention(inp, wl, threads=max(1, os.cpu_count() or 1))
    assert_within(got, ref, wl.tol, "prefill C5 full")


# ------------------------------------------------------ partial / combine --

def test_decode_partial_matches_oracle_splits():
    inp, meta = problem(B=2, Hq=8, Hkv=2, D=128, P=32, lens=(300, 70), dt="f16", num_pages=20,
                        seed=91)
    p = params_of(inp, meta, num_splits=4)
    S, tok = ops.decode_plan(p)
    d = ops.device_inputs(inp, "f16")
    ml = torch.empty((2, 8, S, 2), dtype=torch.float32, device="cuda")
    acc = torch.full((2, 8, S, 128), float("nan"), dtype=torch.float32, device="cuda")
    ops.decode_partial(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                       d["context_lens"], ml, acc, S)
    torch.cuda.synchronize()
    ml, acc = ml.cpu().numpy(), acc.cpu().numpy()
    for s in range(2):
        for h in range(8):
            for i in range(S):
                m_ref, l_ref, acc_ref = oracle.split_partial(inp, s, h, i * tok, (i + 1) * tok, **meta)
                if m_ref == -np.inf:
                    assert ml[s, h, i, 0] == -np.inf and ml[s, h, i, 1] == 0
                    continue
                assert abs(ml[s, h, i, 0] - m_ref) < 1e-4 * max(1, abs(m_ref))
                assert abs(ml[s, h, i, 1] - l_ref) <= 1e-3 * l_ref
                np.testing.assert_allclose(acc[s, h, i], acc_ref, rtol=0, atol=2e-3 * l_ref)


def test_combine_matches_oracle():
    rng = np.random.default_rng(3)
    B, Hq, S, D = 3, 5, 9, 64
    m = rng.normal(0, 4, size=(B, Hq, S)).astype(np.float32)
    m[0, 0, 3:] = -np.inf
    m[1, 2, :] = -np.inf
    l = rng.uniform(1, 50, size=(B, Hq, S)).astype(np.float32)
    l[m == -np.inf] = 0
    acc = rng.normal(0, 10, size=(B, Hq, S, D)).astype(np.float32)
    ml = np.stack([m, l], axis=-1)
    p = ops.make_params(num_seqs=B, num_q_heads=Hq, num_kv_heads=1, head_dim=D, page_size=16,
                        num_pages=1, max_blocks_per_seq=1, max_context_len=16, dtype="f32")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ops.combine(p, torch.from_numpy(ml).cuda(), torch.from_numpy(acc).cuda(), S, out)
    got = out.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            ref = oracle.combine(m[b, h].astype(np.float64), l[b, h], acc[b, h])
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-5, atol=1e-5)
    assert np.array_equal(got[1, 2], np.zeros(D))


def test_combine_splits_per_sequence():
    """splits_per_seq gives each sequence its own split count: sequence b
    merges its first S_b splits (minfer doc 71, Excerpt F: idle splits are
    weighted to zero); the splits past S_b hold NaN and are never read; S_b
    = 0 writes zeros and counts above max_splits are clamped."""
    rng = np.random.default_rng(4)
    B, Hq, S, D = 5, 4, 40, 128
    counts = np.array([1, 40, 0, 33, 77], dtype=np.int32)
    m = rng.normal(0, 3, size=(B, Hq, S)).astype(np.float32)
    m[3, 1, 5:9] = -np.inf
    l = rng.uniform(1, 50, size=(B, Hq, S)).astype(np.float32)
    l[m == -np.inf] = 0
    acc = rng.normal(0, 10, size=(B, Hq, S, D)).astype(np.float32)
    for b in range(B):
        n = min(max(int(counts[b]), 0), S)
        m[b, :, n:] = np.nan
        l[b, :, n:] = np.nan
        acc[b, :, n:] = np.nan
    ml = np.stack([m, l], axis=-1)
    p = ops.make_params(num_seqs=B, num_q_heads=Hq, num_kv_heads=1, head_dim=D, page_size=16,
                        num_pages=1, max_blocks_per_seq=1, max_context_len=16, dtype="f32")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ops.combine(p, torch.from_numpy(ml).cuda(), torch.from_numpy(acc).cuda(), S, out,
                splits_per_seq=torch.from_numpy(counts).cuda())
    got = out.cpu().numpy()
    for b in range(B):
        n = min(max(int(counts[b]), 0), S)
        for h in range(Hq):
            if n == 0:
                assert np.array_equal(got[b, h], np.zeros(D))
                continue
            ref = oracle.combine(m[b, h, :n].astype(np.float64), l[b, h, :n], acc[b, h, :n])
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------- invariances --

def test_permuted_pages_bitwise_identical():
    """Paging moves storage, not arithmetic: the same logical data behind a
    permuted block table gives identical bits (crucible README)."""
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=32, lens=(900, 33, 1), dt="bf16",
                        num_pages=40, shuffle=False, seed=31)
    base, _ = gpu_decode(inp, meta)
    basep, _ = gpu_prefill(dict(inp), meta)
    perm = np.random.default_rng(8).permutation(40)
    k2, v2 = np.empty_like(inp["k_cache"]), np.empty_like(inp["v_cache"])
    k2[perm], v2[perm] = inp["k_cache"], inp["v_cache"]
    bt = inp["block_tables"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved = dict(inp, k_cache=k2, v_cache=v2, block_tables=bt)
    assert bitwise_equal(gpu_decode(moved, meta)[0], base)
    assert bitwise_equal(gpu_prefill(moved, meta)[0], basep)


def test_run_to_run_bitwise_deterministic():
    wl = workloads.C4
    inp = wl.make_inputs()
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    a, _ = gpu_decode(inp, meta, deterministic=1)
    for _ in range(3):
        assert bitwise_equal(gpu_decode(inp, meta, deterministic=1)[0], a)


def test_poisoned_unread_memory_changes_nothing():
    """NaN in unreferenced pages and in slots past each sequence's length
    must not reach the output (crucible results: future poisoning)."""
    inp, meta = problem(B=4, Hq=8, Hkv=2, D=64, P=16, lens=(1, 15, 17, 200), dt="f16",
                        num_pages=30, seed=41)
    base, _ = gpu_decode(inp, meta)
    pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    used = set(int(x) for x in inp["block_tables"].reshape(-1) if x >= 0)
    for pg in range(30):
        if pg not in used:
            pois["k_cache"][pg] = np.nan
            pois["v_cache"][pg] = np.nan
    for s, L in enumerate(inp["context_lens"]):
        last = inp["block_tables"][s][(L - 1) // 16]
        if L % 16:
            pois["k_cache"][last, L % 16:] = np.nan
            pois["v_cache"][last, L % 16:] = np.nan
    got, status = gpu_decode(pois, meta)
    assert status == 0 and bitwise_equal(got, base)


def test_prefill_row_independent_of_later_rows():
    """Changing the K/V of chunk positions after row r leaves row r's bits."""
    inp, meta = problem(B=1, Hq=8, Hkv=1, D=128, P=32, lens=(200,), qlens=(64,), dt="bf16",
                        num_pages=10, seed=51)
    base, _ = gpu_prefill(inp, meta)
    pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    r = 20
    for j in range(136 + r + 1, 200):
        pg = inp["block_tables"][0][j // 32]
        pois["k_cache"][pg, j % 32] = inputs.round_to(np.array([30.0]), "bf16")[0]
        pois["v_cache"][pg, j % 32] = inputs.round_to(np.array([-50.0]), "bf16")[0]
    got, _ = gpu_prefill(pois, meta)
    assert bitwise_equal(got[: r + 1], base[: r + 1])


def test_prefill_poisoned_unread_memory_changes_nothing():
    """Prefill twin of the decode poisoning test: NaN in unreferenced pages and
    in the slots past each context in its last page never reach the output."""
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=32, lens=(45, 200, 97), qlens=(45, 20, 60),
                        dt="bf16", num_pages=16, seed=43)
    base, st0 = gpu_prefill(inp, meta)
    pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    used = set(int(x) for x in inp["block_tables"].reshape(-1) if x >= 0)
    nan = np.uint16(0x7FC0)  # bf16 quiet NaN (storage bits)
    for pg in range(16):
        if pg not in used:
            pois["k_cache"][pg] = nan
            pois["v_cache"][pg] = nan
    for s, L in enumerate(inp["context_lens"]):
        last = inp["block_tables"][s][(L - 1) // 32]
        if L % 32:
            pois["k_cache"][last, L % 32:] = nan
            pois["v_cache"][last, L % 32:] = nan
    got, status = gpu_prefill(pois, meta)
    assert st0 == 0 and status == 0 and bitwise_equal(got, base)
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL["bf16"], "poisoned")


def test_prefill_bad_page_flags_and_skips():
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=128, P=32, lens=(300, 300), qlens=(40, 40),
                        dt="bf16", num_pages=20, seed=65)
    bad = dict(inp, block_tables=inp["block_tables"].copy())
    bad["block_tables"][1, 2] = 5000  # outside the pool
    got, status = gpu_prefill(bad, meta)
    assert status == ops.PA_DEV_BAD_PAGE
    assert np.isfinite(got).all()
    ref = oracle.attention(inp, threads=THREADS, **meta)
    assert_within(got[:40], ref[:40], TOL["bf16"], "unaffected sequence")


def test_prefill_bad_length_flags_and_zeroes():
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=128, P=32, lens=(64, 64), qlens=(32, 32),
                        dt="bf16", num_pages=8, seed=67)
    bad = dict(inp, context_lens=np.array([64, 10], dtype=np.int32))  # L < chunk rows
    got, status = gpu_prefill(bad, meta)
    assert status == ops.PA_DEV_BAD_LEN
    assert np.array_equal(got[32:], np.zeros_like(got[32:]))
    assert_within(got[:32], oracle.attention(inp, threads=THREADS, **meta)[:32], TOL["bf16"], "ok seq")


# ---------------------------------------------------------- device errors --

def test_bad_page_flags_and_skips():
    inp, meta = problem(B=2, Hq=4, Hkv=1, D=64, P=16, lens=(40, 40), dt="f32", num_pages=8,
                        seed=61)
    bad = dict(inp, block_tables=inp["block_tables"].copy())
    bad["block_tables"][1, 1] = 1000  # outside the pool
    got, status = gpu_decode(bad, meta)
    assert status == ops.PA_DEV_BAD_PAGE
    assert np.isfinite(got).all()
    ref = oracle.attention(inp, **meta)
    assert_within(got[0], ref[0], TOL["f32"], "unaffected sequence")


def test_bad_length_flags_and_zeroes():
    inp, meta = problem(B=2, Hq=4, Hkv=1, D=64, P=16, lens=(40, 40), dt="f32", num_pages=8,
                        seed=63)
    bad = dict(inp, context_lens=np.array([40, 10_000], dtype=np.int32))
    got, status = gpu_decode(bad, meta)
    assert status == ops.PA_DEV_BAD_LEN
    assert np.array_equal(got[1], np.zeros_like(got[1]))
    bad0 = dict(inp, context_lens=np.array([0, 40], dtype=np.int32))
    got, status = gpu_decode(bad0, meta)
    assert status == ops.PA_DEV_BAD_LEN and np.array_equal(got[0], np.zeros_like(got[0]))


# ------------------------------------------------------------ CUDA graphs --

def test_graph_replay_with_new_lengths():
    """Grids depend on host params only, so a captured call replays with new
    device lengths (crucible README: split count fixed at capacity)."""
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=128, P=32, lens=(1000, 1000), dt="bf16",
                        num_pages=70, seed=71)
    inp["context_lens"] = np.array([700, 300], dtype=np.int32)
    p = params_of(inp, meta)
    d = ops.device_inputs(inp, "bf16")
    out = torch.empty((2, 16, 128), dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(ops.decode_workspace_size(p), 1), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
               out=out, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   out=out, workspace=ws, stream=s)
    for lens in ((700, 300), (5, 1000), (1, 1)):
        d["context_lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.attention(dict(inp, context_lens=np.array(lens, dtype=np.int32)), **meta)
        assert_within(out.cpu().numpy(), ref, TOL["bf16"], f"replay {lens}")
