"""Sliding-window decode (pa_params.sliding_window) against the fp64 oracle,
through the C ABI.

A row whose causal end is key e attends keys e - W + 1 ..= e.  Keys before
every row's window are never read: the poisoning test fills them with NaN on
the device and expects the clean oracle's answer.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, inputs, ops, workloads
from helpers import problem, assert_within

pytestmark = pytest.mark.gpu

TOL = {"f32": workloads.TOL_F32, "f16": workloads.TOL_16, "bf16": workloads.TOL_16}
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def params(inp, meta, **kw):
    bt = inp["block_tables"]
    P = meta["page_size"]
    return ops.make_params(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                           num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"], page_size=P,
                           num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                           max_context_len=bt.shape[1] * P, scale=meta["scale"], dtype=meta["q_dtype"],
                           kv_dtype=meta["kv_dtype"], **kw)


def run(inp, meta, **kw):
    p = params(inp, meta, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


CASES = [
    # B, Hq, Hkv, D, P, lens, W, dtype
    (5, 16, 4, 128, 32, (1, 31, 33, 700, 2047), 1, "bf16"),
    (5, 16, 4, 128, 32, (1, 31, 33, 700, 2047), 17, "bf16"),    # inside one page
    (5, 16, 4, 128, 32, (1, 31, 33, 700, 2047), 100, "f16"),    # across pages
    (5, 16, 4, 128, 32, (1, 31, 33, 700, 2047), 5000, "bf16"),  # wider than every context
    (2, 28, 4, 128, 16, (17, 3000), 50, "f16"),                 # G 7, 16-slot pages
    (2, 32, 2, 64, 32, (64, 1500), 300, "bf16"),                # G 16: two column tiles
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-P{c[4]}-W{c[6]}-{c[7]}")
def test_window_decode_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, W, dt = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt,
                        num_pages=sum((L + P - 1) // P for L in lens) + 5, seed=51)
    got, status = run(inp, meta, sliding_window=W)
    assert status == 0
    assert_within(got, oracle.attention(inp, window=W, threads=THREADS, **meta), TOL[dt], f"W={W}")


def test_window_with_several_rows():
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=32, lens=(40, 333, 1200), qlens=(3, 3, 3), dt="bf16",
                        num_pages=60, seed=52)
    got, status = run(inp, meta, sliding_window=40, decode_q_rows=3)
    assert status == 0
    assert_within(got, oracle.attention(inp, window=40, threads=THREADS, **meta), TOL["bf16"], "W=40 T=3")


def test_window_with_append():
    """The appended token is the last key of its own window."""
    inp, meta = problem(B=2, Hq=16, Hkv=4, D=128, P=32, lens=(70, 900), dt="f16", num_pages=40, seed=53)
    k_new, v_new = inputs.make_append_rows(num_seqs=2, num_kv_heads=4, head_dim=128, kv_dtype="f16", seed=54)
    expect = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    for b, L in enumerate(inp["context_lens"]):
        pg, slot = inp["block_tables"][b, (L - 1) // 32], (L - 1) % 32
        expect["k_cache"][pg, slot] = k_new[b]
        expect["v_cache"][pg, slot] = v_new[b]
    p = params(inp, meta, sliding_window=64)
    d = ops.device_inputs(inp, "f16")
    out = ops.decode_append(p, d["q"], ops.to_device(k_new, "f16"), ops.to_device(v_new, "f16"),
                            d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    torch.cuda.synchronize()
    assert_within(out.cpu().numpy(), oracle.attention(expect, window=64, threads=THREADS, **meta),
                  TOL["f16"], "append W=64")


def test_keys_before_the_window_are_never_read():
    """NaN in every K and V row before the windows (whole pages and the head
    of the first window page) leaves the result equal to the clean oracle's."""
    W = 45
    inp, meta = problem(B=3, Hq=16, Hkv=4, D=128, P=32, lens=(50, 700, 2000), dt="bf16", num_pages=90,
                        seed=55)
    ref = oracle.attention(inp, window=W, threads=THREADS, **meta)
    k, v = inp["k_cache"].copy(), inp["v_cache"].copy()
    for b, L in enumerate(inp["context_lens"]):
        for j in range(L - W):
            pg = inp["block_tables"][b, j // 32]
            k[pg, j % 32] = np.uint16(0x7FC0)
            v[pg, j % 32] = np.uint16(0x7FC0)
    got, status = run(dict(inp, k_cache=k, v_cache=v), meta, sliding_window=W)
    assert status == 0
    assert_within(got, ref, TOL["bf16"], "poisoned pre-window keys")


def test_window_unsupported_paths_are_rejected():
    inp, meta = problem(B=1, Hq=4, Hkv=2, D=64, P=16, lens=(40,), dt="f32", num_pages=4, seed=56)
    with pytest.raises(ops.PaError):
        run(inp, meta, sliding_window=8)  # fp32 K/V
    inp, meta = problem(B=1, Hq=4, Hkv=2, D=128, P=32, lens=(40,), dt="bf16", num_pages=4, seed=57)
    with pytest.raises(ops.PaError):
        run(inp, meta, sliding_window=8, num_splits=2)  # fixed split plan


def test_window_full_size_ragged_batch():
    """The ragged 16-sequence decode batch with a 1024-key window."""
    wl = workloads.BY_NAME["ragged_b16_32x8_d128"]
    inp = wl.make_inputs()
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, status = run(inp, meta, sliding_window=1024)
    assert status == 0
    assert_within(got, oracle.attention(inp, window=1024, threads=THREADS, **meta), TOL["bf16"], "W=1024")
