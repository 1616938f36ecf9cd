"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

None of these compares the oracle with itself: each expected value is a
closed form, a value printed on the pages (``tests/golden``), a library
routine, an independently written brute-force path, or an invariance the
definition implies.  ``test_planted_mistakes_are_caught`` shows that each
plausible mistake planted in the oracle fails at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
from oracle import dense
from paged_kv_gqa_02_gb300 import inputs, workloads
from helpers import problem, dense_ref, f64, bitwise_equal, within, assert_within

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def kv_vec(inp, meta, pool, s, j, g):
    """float64 vector of logical key j, kv head g of sequence s (by table)."""
    P = meta["page_size"]
    page = inp["block_tables"][s][j // P]
    return inputs.as_float64(inp[pool][page, j % P, g], meta["kv_dtype"])


# ---------------------------------------------------------------- pins ----

def pin_length_one():
    """L = 1: the only weight is 1, so out = v_0 exactly (any q, k)."""
    ok = True
    for dt in ("f32", "f16", "bf16"):
        inp, meta = problem(B=3, Hq=6, Hkv=3, D=16, P=4, lens=(1, 1, 1), dt=dt, seed=3)
        out = oracle.attention(inp, **meta)
        for s in range(3):
            for h in range(6):
                ok &= bool(np.array_equal(out[s, h], kv_vec(inp, meta, "v_cache", s, 0, h // 2)))
    return ok


def pin_uniform_keys():
    """All keys of a (seq, kv head) equal: every weight equal, out = mean_j v_j."""
    inp, meta = problem(B=2, Hq=8, Hkv=2, D=16, P=4, lens=(13, 6), dt="f32", seed=5)
    k = inp["k_cache"]
    for s, L in enumerate(inp["context_lens"]):
        for g in range(2):
            ref = k[inp["block_tables"][s][0], 0, g].copy()
            for j in range(L):
                k[inp["block_tables"][s][j // 4], j % 4, g] = ref
    out = oracle.attention(inp, **meta)
    ok = True
    for s, L in enumerate(inp["context_lens"]):
        for h in range(8):
            mean = np.mean([kv_vec(inp, meta, "v_cache", s, j, h // 4) for j in range(L)], axis=0)
            ok &= bool(np.abs(out[s, h] - mean).max() < 1e-13)
    return ok


def pin_constant_v_per_group():
    """V = g+1 on every key of kv head g: out = g+1 for every q head of group g
    (the GQA grouping h -> h / (Hq/Hkv) of the pages' mapping)."""
    inp, meta = problem(B=2, Hq=12, Hkv=3, D=8, P=4, lens=(9, 17), dt="f32", seed=7)
    for g in range(3):
        inp["v_cache"][:, :, g, :] = g + 1.0
    out = oracle.attention(inp, **meta)
    want = np.repeat(np.arange(1.0, 4.0), 4)[None, :, None]
    return bool(np.abs(out - want).max() < 1e-13)


def pin_two_keys_closed_form():
    """Two keys with scores a*scale and 0 by construction:
    out = sigmoid(a*scale) v0 + (1 - sigmoid(a*scale)) v1."""
    inp, meta = problem(B=1, Hq=2, Hkv=1, D=4, P=2, lens=(2,), dt="f32", seed=9, scale=0.75)
    a = [1.5, -2.25]
    for h in range(2):
        inp["q"][0, h] = [a[h], 0, 0, 0]
    page = inp["block_tables"][0][0]
    inp["k_cache"][page, 0, 0] = [1, 0, 0, 0]
    inp["k_cache"][page, 1, 0] = [0, 1, 0, 0]
    out = oracle.attention(inp, **meta)
    v0, v1 = (inputs.as_float64(inp["v_cache"][page, j, 0], "f32") for j in (0, 1))
    ok = True
    for h in range(2):
        sig = 1.0 / (1.0 + math.exp(-a[h] * 0.75))
        ok &= bool(np.abs(out[0, h] - (sig * v0 + (1 - sig) * v1)).max() < 1e-14)
    return ok


def pin_dominant_key():
    """q parallel to one key and a scale large enough that scores pass the
    double exp range (~709): the max subtraction keeps it finite and the
    result is v of that key."""
    inp, meta = problem(B=1, Hq=1, Hkv=1, D=8, P=4, lens=(11,), dt="f32", seed=11, scale=400.0)
    jstar = 6
    kstar = kv_vec(inp, meta, "k_cache", 0, jstar, 0)
    inp["q"][0, 0] = (kstar / np.linalg.norm(kstar) * 4).astype(np.float32)
    out = oracle.attention(inp, **meta)
    return bool(np.abs(out[0, 0] - kv_vec(inp, meta, "v_cache", 0, jstar, 0)).max() < 1e-6)


def pin_dense_agreement(cases=None):
    """Brute force (dense materialisation + numpy) on tiny shapes, decode and
    prefill, every dtype and page size."""
    rng = np.random.default_rng(1234)
    ok = True
    for c in range(cases or 24):
        P = int(rng.choice([4, 16, 32]))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 3, 4, 5, 7, 8]))
        D = int(rng.choice([8, 16, 64, 128]))
        B = int(rng.integers(1, 4))
        lens = [int(x) for x in rng.integers(1, 71, size=B)]
        qlens = [1 if c % 2 == 0 else int(rng.integers(1, L + 1)) for L in lens]
        dt = ("f32", "f16", "bf16")[c % 3]
        inp, meta = problem(B=B, Hq=G * Hkv, Hkv=Hkv, D=D, P=P, lens=lens, qlens=qlens, dt=dt,
                            num_pages=sum((L + P - 1) // P for L in lens) + 5, seed=100 + c)
        ok &= bool(np.abs(oracle.attention(inp, **meta) - dense_ref(inp, meta)).max() < 1e-12)
    return ok


def pin_window_one():
    """Sliding window of 1: a row sees only its own position, so out is that
    key's v exactly, for decode and prefill rows and every dtype."""
    ok = True
    for dt in ("f32", "f16", "bf16"):
        inp, meta = problem(B=2, Hq=6, Hkv=3, D=16, P=4, lens=(9, 14), qlens=(1, 5), dt=dt, seed=41)
        out = oracle.attention(inp, window=1, **meta)
        for s in range(2):
            L, r0, r1 = int(inp["context_lens"][s]), int(inp["cu_q_lens"][s]), int(inp["cu_q_lens"][s + 1])
            for r in range(r0, r1):
                end = L - (r1 - r0) + (r - r0)
                for h in range(6):
                    ok &= bool(np.array_equal(out[r, h], kv_vec(inp, meta, "v_cache", s, end, h // 2)))
    return ok


def pin_window_dense_agreement():
    """Windowed attention against the dense brute force with the same window
    mask, on random tiny shapes, decode and prefill rows."""
    rng = np.random.default_rng(4321)
    ok = True
    for c in range(12):
        P = int(rng.choice([4, 16]))
        Hkv, G = int(rng.integers(1, 3)), int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        lens = [int(x) for x in rng.integers(1, 60, size=B)]
        qlens = [1 if c % 2 == 0 else int(rng.integers(1, L + 1)) for L in lens]
        W = int(rng.integers(1, 40))
        inp, meta = problem(B=B, Hq=G * Hkv, Hkv=Hkv, D=16, P=P, lens=lens, qlens=qlens,
                            dt=("f32", "bf16")[c % 2], num_pages=sum((L + P - 1) // P for L in lens) + 3,
                            seed=300 + c)
        q, k, v = f64(inp, meta)
        ref = dense.attention(q, k, v, inp["block_tables"], inp["context_lens"], inp["cu_q_lens"],
                              meta["num_q_heads"], meta["num_kv_heads"], meta["page_size"], meta["scale"],
                              window=W)
        ok &= bool(np.abs(oracle.attention(inp, window=W, **meta) - ref).max() < 1e-12)
    return ok


def pin_window_wider_than_context():
    """A window at least as long as the context changes nothing (bitwise)."""
    inp, meta = problem(B=2, Hq=4, Hkv=2, D=16, P=8, lens=(37, 12), qlens=(1, 3), dt="f16", seed=43)
    return bitwise_equal(oracle.attention(inp, window=37, **meta), oracle.attention(inp, **meta))


def pin_page_boundaries():
    ok = True
    for P, lens in ((32, (1, 31, 32, 33, 63, 64, 65)), (16, (1, 15, 16, 17, 1023, 1024))):
        inp, meta = problem(B=len(lens), Hq=4, Hkv=2, D=16, P=P, lens=lens, dt="bf16", seed=P)
        ok &= bool(np.abs(oracle.attention(inp, **meta) - dense_ref(inp, meta)).max() < 1e-12)
    return ok


def pin_causal_positions():
    """Sum over query rows of the keys attended equals the crucible results'
    printed 'sum of causal positions' for each microbenchmark shape."""
    ok = True
    for name, rows, offs, want in read_causal_golden():
        lens = [o + t for o, t in zip(offs, rows)]
        inp, meta = problem(B=len(rows), Hq=1, Hkv=1, D=1, P=16, lens=lens, qlens=rows,
                            dt="f32", seed=1)
        _, keys = oracle.attention(inp, return_keys=True, **meta)
        ok &= keys == want
    return ok


def pin_outliers():
    """The minfer doc 71 outlier recipe (|q| ~ 57, |v| ~ 144) stays finite and
    matches brute force."""
    inp, meta = problem(B=1, Hq=5, Hkv=1, D=128, P=32, lens=(300,), dt="f32", seed=13)
    i = np.arange(inp["q"].size)
    inp["q"].reshape(-1)[:] = (((i * 37) % 19) / 5 - 1.9) * 30
    iv = np.arange(inp["v_cache"].size)
    inp["v_cache"].reshape(-1)[:] = (((iv * 57) % 11) / 3 - 1.8) * 80
    out = oracle.attention(inp, **meta)
    return bool(np.isfinite(out).all() and np.abs(out - dense_ref(inp, meta)).max() < 1e-9)


PINS = [pin_length_one, pin_uniform_keys, pin_constant_v_per_group, pin_two_keys_closed_form,
        pin_dominant_key, pin_dense_agreement, pin_page_boundaries, pin_causal_positions,
        pin_outliers, pin_window_one, pin_window_dense_agreement, pin_window_wider_than_context]


def read_causal_golden():
    out = []
    with open(os.path.join(GOLDEN, "crucible_causal_positions.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, rows, offs, want = (x.strip() for x in line.split(";"))

            def expand(spec):
                if "*" in spec:
                    v, n = spec.split("*")
                    return [int(v)] * int(n)
                return [int(x) for x in spec.split(",")]
            out.append((name, expand(rows), expand(offs), int(want)))
    return out


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    assert pin()


def test_planted_mistakes_are_caught():
    """Each deliberate mistake planted in the oracle (interleaved GQA mapping,
    off-by-one causal end, shifted slot, score sign, missing max shift,
    reversed V index, wrong normaliser, window one key too wide) fails at
    least one pin."""
    try:
        for m in range(1, 9):
            oracle.set_mutation(m)
            results = []
            for pin in PINS:
                try:
                    results.append(bool(pin()))
                except (ValueError, AssertionError, FloatingPointError):
                    results.append(False)
            assert not all(results), f"mutation {m} passed every pin"
    finally:
        oracle.set_mutation(0)
    assert all(p() for p in PINS[:3])


# -------------------------------------------------------- invariances ----

def test_permuted_table_matches_identity_bitwise():
    """Paging moves storage, not arithmetic (crucible README, paged KV
    correctness): the same data behind a permuted table gives identical bits."""
    inp, meta = problem(B=3, Hq=8, Hkv=2, D=32, P=16, lens=(70, 33, 1), dt="f16",
                        num_pages=12, shuffle=False, seed=21)
    base = oracle.attention(inp, **meta)
    perm = np.random.default_rng(5).permutation(12)
    k2 = np.empty_like(inp["k_cache"])
    v2 = np.empty_like(inp["v_cache"])
    k2[perm] = inp["k_cache"]
    v2[perm] = inp["v_cache"]
    bt = inp["block_tables"].copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved = dict(inp, k_cache=k2, v_cache=v2, block_tables=bt)
    assert bitwise_equal(oracle.attention(moved, **meta), base)


def test_future_poisoning_leaves_rows_unchanged():
    """Keys after a row's causal end, tail slots of the last page, unreferenced
    pages and unused table entries are never read."""
    inp, meta = problem(B=2, Hq=4, Hkv=2, D=16, P=8, lens=(29, 20), qlens=(9, 4), dt="f32",
                        num_pages=10, seed=23)
    base = oracle.attention(inp, **meta)
    # poison: unreferenced pages and the tail of each last page
    pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    used = set(int(x) for x in inp["block_tables"].reshape(-1) if x >= 0)
    for p in range(10):
        if p not in used:
            pois["k_cache"][p] = np.nan
            pois["v_cache"][p] = np.nan
    for s, L in enumerate(inp["context_lens"]):
        last = inp["block_tables"][s][(L - 1) // 8]
        pois["k_cache"][last, L % 8 or 8:] = np.nan
        pois["v_cache"][last, L % 8 or 8:] = np.nan
    assert bitwise_equal(oracle.attention(pois, **meta), base)
    # row r of seq 0 (start = 20) must not see keys > 20 + r
    r = 3
    row_pois = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    for j in range(20 + r + 1, 29):
        pg = inp["block_tables"][0][j // 8]
        row_pois["k_cache"][pg, j % 8] = 1e30
        row_pois["v_cache"][pg, j % 8] = np.nan
    got = oracle.attention_one(row_pois, r, 1, **meta)
    assert bitwise_equal(got, base[r, 1])


def test_keys_before_the_window_are_never_read():
    """NaN in every key and value a row's window excludes leaves its output
    unchanged (bitwise): the window is a read bound, not a mask."""
    inp, meta = problem(B=1, Hq=4, Hkv=2, D=16, P=8, lens=(40,), qlens=(1,), dt="f32", seed=47)
    W = 13
    base = oracle.attention(inp, window=W, **meta)
    k, v = inp["k_cache"].copy(), inp["v_cache"].copy()
    for j in range(40 - W):
        pg = inp["block_tables"][0][j // 8]
        k[pg, j % 8] = np.nan
        v[pg, j % 8] = np.nan
    poisoned = dict(inp, k_cache=k, v_cache=v)
    assert bitwise_equal(oracle.attention(poisoned, window=W, **meta), base)


def test_prefill_row_equals_decode_at_that_length():
    """Chunk row r attends the same keys as a decode of length start + r + 1."""
    inp, meta = problem(B=1, Hq=6, Hkv=2, D=16, P=4, lens=(23,), qlens=(7,), dt="bf16", seed=25)
    full = oracle.attention(inp, **meta)
    for r in range(7):
        dec = dict(inp, q=inp["q"][r:r + 1].copy(),
                   context_lens=np.array([16 + r + 1], dtype=np.int32),
                   cu_q_lens=np.array([0, 1], dtype=np.int32))
        assert bitwise_equal(oracle.attention(dec, **meta)[0], full[r])


def test_split_combine_equals_full():
    """Splitting keys into ranges, summarising each (m, l, acc) and combining
    gives the single-pass result (crucible README, split-position attention);
    empty splits (m = -inf) get weight 0."""
    inp, meta = problem(B=2, Hq=6, Hkv=3, D=32, P=16, lens=(100, 37), dt="f16", seed=27)
    full = oracle.attention(inp, **meta)
    for s, L in enumerate(inp["context_lens"]):
        for h in range(6):
            bounds = [0, 16, 48, 64, 112, 128]
            parts = [oracle.split_partial(inp, s, h, a, b, **meta)
                     for a, b in zip(bounds[:-1], bounds[1:])]
            m = [p[0] for p in parts]
            l = [p[1] for p in parts]
            acc = np.stack([p[2] for p in parts])
            assert any(x == -np.inf for x in m) or L > 112
            np.testing.assert_allclose(oracle.combine(m, l, acc), full[s, h], rtol=0, atol=1e-12)


def test_combine_closed_form():
    """Two splits whose summaries are given: weights 2^(m_i - max m)."""
    m = [3.0, 1.0, -np.inf]
    l = [2.0, 5.0, 0.0]
    acc = np.array([[4.0, -2.0], [10.0, 1.0], [7.0, 7.0]])
    want = (np.array([4.0, -2.0]) * 1 + np.array([10.0, 1.0]) * 0.25) / (2.0 + 5.0 * 0.25)
    np.testing.assert_allclose(oracle.combine(m, l, acc), want, rtol=0, atol=1e-15)
    assert np.array_equal(oracle.combine([-np.inf], [0.0], np.ones((1, 2))), [0.0, 0.0])


def test_rejects_bad_metadata():
    inp, meta = problem(B=1, Hq=2, Hkv=1, D=4, P=4, lens=(6,), dt="f32", seed=29)
    bad = dict(inp, block_tables=inp["block_tables"].copy())
    bad["block_tables"][0, 1] = 99
    with pytest.raises(ValueError):
        oracle.attention(bad, **meta)
    with pytest.raises(ValueError):
        oracle.attention(dict(inp, context_lens=np.array([0], dtype=np.int32)), **meta)


# ------------------------------------------------- library / printed pins --

def test_upcast_matches_numpy_for_every_bit_pattern():
    """The oracle's binary16/bfloat16 decoders equal numpy's conversions on all
    65,536 bit patterns (NaNs compared as NaN)."""
    bits = np.arange(65536, dtype=np.uint16)
    for dt, ref in (("f16", bits.view(np.float16).astype(np.float64)),
                    ("bf16", inputs.bf16_bits_to_f32(bits).astype(np.float64))):
        got = np.array([oracle.upcast(dt, bits, i) for i in range(0, 65536, 1)])
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def test_byte_ledgers_match_pages():
    rows = {}
    with open(os.path.join(GOLDEN, "byte_ledgers.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, _, val = (x.strip() for x in line.split(";"))
                rows[name] = float(val)
    c3 = workloads.C3
    assert c3.kv_bytes() == rows["minfer_14b_L3254"]
    assert round(c3.kv_bytes() / 1e6, 1) == rows["minfer_14b_L3254_rounded_MB"]
    c1 = workloads.C1
    per_key_per_kv_head = 2 * c1.head_dim * c1.elt(c1.kv_dtype)
    assert per_key_per_kv_head == rows["crucible_per_kv_head_per_key"]
    assert per_key_per_kv_head * c1.num_q_heads == rows["crucible_per_q_head_per_key"]
    for name, rows_, offs, want in read_causal_golden():
        if name == "16x16":
            assert want == rows["crucible_16x16_S"]
        if name == "4x256":
            assert want == rows["crucible_4x256_S"]


def test_workload_visible_keys_match_pages():
    """The workload byte/flop accounting uses the same causal bound."""
    for name, rows, offs, want in read_causal_golden():
        w = workloads.Workload(name=name, kind="prefill", num_seqs=len(rows), num_q_heads=1,
                               num_kv_heads=1, head_dim=1, page_size=16, q_dtype="f32",
                               kv_dtype="f32", context_lens=tuple(o + t for o, t in zip(offs, rows)),
                               q_lens=tuple(rows), num_pages=1, max_blocks_per_seq=1,
                               shuffle=False, scale=1.0)
        assert w.visible_keys() == want


def test_named_packed_workloads_are_the_pages_shapes():
    """The bench's packed-prefill workloads are the pages' 16x16 and 4x256
    shapes: their causal bound is the printed sum of causal positions."""
    want = {name: s for name, _, _, s in read_causal_golden()}
    for wl in (workloads.PACK_F32, workloads.PACK_BF16):
        assert wl.visible_keys() == want["16x16"]
    for wl in (workloads.PACK4_F32, workloads.PACK4_BF16):
        assert wl.visible_keys() == want["4x256"]
        assert wl.flops() == 4 * want["4x256"] * wl.num_q_heads * wl.head_dim


def test_generator_lengths_and_stream():
    """The ragged batch lengths: forced 1/31/32/33 then seeded draws."""
    L = inputs.ragged_lengths(inputs.DEFAULT_SEED, 12)
    assert L[:4] == [1, 31, 32, 33]
    assert all(1 <= x <= 4096 for x in L)
    assert sum((x + 31) // 32 for x in L) <= 4096
    g = inputs.SplitMix64(0)
    # first output of splitmix64 seeded 0 (published test value of the mixer)
    assert g.next() == 0xE220A8397B1DCDAF


def test_comparator_detects_single_ulp_and_tolerance_breaks():
    """Comparator self-test (vllm.cpp PR #383, 'Comparator self-test'):
    corrupting offsets 5, 1024 and 2047 of 2048 elements is detected."""
    rng = np.random.default_rng(0)
    ref = rng.standard_normal(2048).astype(np.float32)
    for off in (5, 1024, 2047):
        bad = ref.copy()
        bad[off] = np.nextafter(bad[off], np.float32(np.inf))
        assert not bitwise_equal(bad, ref)
        bad2 = ref.astype(np.float64)
        bad2[off] += 3e-3
        assert not within(bad2, ref, {"abs": 2e-3, "rel": 1e-2, "rel_floor": 1e-2})
    assert bitwise_equal(ref.copy(), ref) and within(ref, ref, {"abs": 0.0})
