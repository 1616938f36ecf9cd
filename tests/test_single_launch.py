"""Counted single-launch decode (pa_params.decode_form = PA_FORM_COUNTED):
the split-KV kernel finishes every unit itself.

16-bit K/V with automatic splits, head_dim <= 128 and at most 8 MMA columns
(query rows x q heads per kv head) then run pa_decode as one kernel: each CTA
merges its warps' pieces, and the last CTA to leave a piece of a unit,
counted on an arrival counter at the head of the workspace, merges that
unit's CTA pieces in ascending CTA order (split-KV combine: crucible README,
"Split-position attention").  The counters must be zero before the first
call on a workspace and every call leaves them zero.
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

TOL = workloads.TOL_16
THREADS = max(1, min(16, os.cpu_count() or 1))
COUNTER_BYTES = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def _params(inp, meta, **kw):
    bt = inp["block_tables"]
    args = dict(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"],
                page_size=meta["page_size"], num_pages=int(inp["num_pages"]),
                max_blocks_per_seq=bt.shape[1], max_context_len=bt.shape[1] * meta["page_size"],
                scale=meta["scale"], dtype=meta["q_dtype"], kv_dtype=meta["kv_dtype"],
                decode_form=ops.PA_FORM_COUNTED)
    args.update(kw)
    return ops.make_params(**args)


def _run(inp, meta, ws=None, out=None, **kw):
    p = _params(inp, meta, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     out=out, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


def _counters_zero(ws) -> bool:
    return int(torch.count_nonzero(ws[:COUNTER_BYTES]).item()) == 0


SHAPES = [
    # B, Hq, Hkv, D, P, lens, dtype
    (16, 32, 8, 128, 32, (1, 31, 32, 33, 2721, 2442, 805, 3081, 278, 2616, 3061, 2801, 3732, 3150,
                          42, 2132), "bf16"),
    (1, 40, 8, 128, 32, (3254,), "f16"),
    (3, 28, 4, 128, 32, (1641, 7, 900), "f16"),
    (40, 16, 4, 64, 16, tuple(1 + (i * 997) % 700 for i in range(40)), "bf16"),
    (2, 8, 1, 128, 32, (20000, 3), "bf16"),
]


def test_kernels_per_call():
    """pa_decode_kernels: the counted form is one kernel, the pair two, a
    single-split fixed plan one, and the fp32 append adds its scatter."""
    inp, meta = problem(B=2, Hq=32, Hkv=8, D=128, P=32, lens=(3000, 40), dt="bf16", num_pages=100, seed=3)
    assert ops.decode_kernels(_params(inp, meta)) == 1
    for form in (ops.PA_FORM_AUTO, ops.PA_FORM_PAIR):
        assert ops.decode_kernels(_params(inp, meta, decode_form=form)) == 2
    assert ops.decode_kernels(_params(inp, meta, decode_phases=1)) == 1
    assert ops.decode_kernels(_params(inp, meta, num_splits=1)) == 1
    assert ops.decode_kernels(_params(inp, meta, num_splits=4)) == 2
    f32, m32 = problem(B=2, Hq=8, Hkv=2, D=64, P=16, lens=(300, 40), dt="f32", num_pages=30, seed=4)
    assert ops.decode_kernels(_params(f32, m32), with_append=True) == 3
    assert ops.decode_kernels(_params(inp, meta, head_dim=96)) == -1


def test_one_workspace_serves_every_shape_and_counters_stay_zero():
    """One zeroed buffer, calls of different sizes in turn: each result
    matches the oracle, and the counter block is zero after every call."""
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for i, (B, Hq, Hkv, D, P, lens, dt) in enumerate(SHAPES):
            npages = sum((L + P - 1) // P for L in lens) + 9
            inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt, num_pages=npages,
                                seed=500 + i)
            p = _params(inp, meta)
            assert ops.decode_workspace_size(p) <= ws.numel()
            got, status = _run(inp, meta, ws=ws)
            assert status == 0
            assert _counters_zero(ws), f"counters left set after shape {i}"
            if rep == 0:
                ref = oracle.attention(inp, threads=THREADS, **meta)
                assert_within(got, ref, TOL, f"shape {i}")


def test_single_launch_matches_the_two_kernel_form():
    """decode_phases 1 then 2 (partial kernel, then combine kernel) and the
    counted single launch agree within the decode tolerance and both match the
    oracle; the single launch is bit-identical run to run."""
    for i, (B, Hq, Hkv, D, P, lens, dt) in enumerate(SHAPES[:3]):
        npages = sum((L + P - 1) // P for L in lens) + 5
        inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt, num_pages=npages,
                            seed=600 + i)
        one, _ = _run(inp, meta)
        assert bitwise_equal(_run(inp, meta)[0], one)
        p = _params(inp, meta)
        d = ops.device_inputs(inp, dt)
        ws = torch.zeros(ops.decode_workspace_size(p), dtype=torch.uint8, device="cuda")
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        for ph in (1, 2):
            p.decode_phases = ph
            ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                       out=out, workspace=ws)
        torch.cuda.synchronize()
        two = out.cpu().numpy()
        ref = oracle.attention(inp, threads=THREADS, **meta)
        assert_within(one, ref, TOL, f"single launch {i}")
        assert_within(two, ref, TOL, f"two kernels {i}")
        assert_within(one, two.astype(np.float64), TOL, f"single vs two kernels {i}")


def test_single_launch_invalid_length_and_page():
    """A sequence with an invalid length is written as zeros with
    PA_DEV_BAD_LEN (no unit exists for it); an out-of-pool page is skipped
    with PA_DEV_BAD_PAGE; the others are unaffected and the counters end at
    zero."""
    lens = (40, 3000, 1, 2000)
    inp, meta = problem(B=4, Hq=16, Hkv=4, D=128, P=32, lens=lens, dt="bf16", num_pages=180,
                        seed=71)
    ref = oracle.attention(inp, threads=THREADS, **meta)
    ws = torch.zeros(ops.decode_workspace_size(_params(inp, meta)), dtype=torch.uint8, device="cuda")
    bad = dict(inp, context_lens=np.array([40, 10_000_000, 1, 0], dtype=np.int32))
    got, status = _run(bad, meta, ws=ws)
    assert status == ops.PA_DEV_BAD_LEN
    assert np.array_equal(got[1], np.zeros_like(got[1])) and np.array_equal(got[3], np.zeros_like(got[3]))
    assert_within(got[[0, 2]], ref[[0, 2]], TOL, "valid sequences beside invalid ones")
    assert _counters_zero(ws)
    badp = dict(inp, block_tables=inp["block_tables"].copy())
    badp["block_tables"][1, 5] = 1 << 20
    got, status = _run(badp, meta, ws=ws)
    assert status == ops.PA_DEV_BAD_PAGE and np.isfinite(got).all()
    assert_within(got[[0, 2, 3]], ref[[0, 2, 3]], TOL, "sequences beside a bad page")
    assert _counters_zero(ws)


def test_one_unit_over_every_cta():
    """One kv head and one long sequence: the unit is split over every CTA of
    the grid, so the last CTA merges ~150 pieces (several load batches)."""
    inp, meta = problem(B=1, Hq=8, Hkv=1, D=128, P=32, lens=(30000,), dt="f16", num_pages=940,
                        seed=81)
    got, status = _run(inp, meta)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL, "one unit over the grid")


def test_device_sm_partition():
    """deterministic = 0 takes the device's SM count for the grid; results
    still match the oracle and repeat bit for bit."""
    B, Hq, Hkv, D, P, lens, dt = SHAPES[0]
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt, num_pages=900, seed=91)
    a, status = _run(inp, meta, deterministic=0)
    assert status == 0
    assert bitwise_equal(_run(inp, meta, deterministic=0)[0], a)
    assert_within(a, oracle.attention(inp, threads=THREADS, **meta), TOL, "device SM count")
