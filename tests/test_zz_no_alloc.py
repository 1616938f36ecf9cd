"""pa_decode_noalloc: decode for callers that cannot allocate device memory
at call time (an engine plugin whose host owns every buffer, a serving loop
that forbids allocation after start-up).  It keeps the split partials in the
library's static device scratch instead of a caller workspace.

This file is named to be collected last: a run that stops at the first
failure has run every other test before this one.  It passes alone in a
fresh process (its first call does the per-device set-up) and after them.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, ops, workloads
from helpers import problem, assert_within, bitwise_equal

pytestmark = pytest.mark.gpu


def _params(inp, meta, **kw):
    bt = inp["block_tables"]
    return ops.make_params(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                           num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"],
                           page_size=meta["page_size"], num_pages=int(inp["num_pages"]),
                           max_blocks_per_seq=bt.shape[1],
                           max_context_len=bt.shape[1] * meta["page_size"], scale=meta["scale"],
                           dtype=meta["q_dtype"], kv_dtype=meta["kv_dtype"], **kw)


def _split_pair(p, d, S):
    """pa_decode_partial then pa_combine on a caller-allocated workspace: the
    two kernels pa_decode_noalloc runs, with the same split plan."""
    B, Hq, D = p.num_seqs, p.num_q_heads, p.head_dim
    ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device="cuda")
    acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ops.decode_partial(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                       d["context_lens"], ml, acc, S)
    ops.combine(p, ml, acc, S, out)
    return out


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    """Two consecutive calls with different batches.  Each is checked three
    ways: against the fp64 oracle at the 16-bit decode tolerance, against
    pa_decode with a caller workspace (another kernel pair) at the same
    tolerance, and bit for bit against the same partial and combine kernels
    run on a caller workspace.  The scratch left by the first call therefore
    does not leak into the second."""
    build.build()
    tol = workloads.TOL_16
    cases = [((1, 31, 32, 33, 2721, 805, 3081, 42), 11), ((700, 1, 4000, 64, 5, 2047, 33, 999), 12)]
    for lens, seed in cases:
        inp, meta = problem(B=8, Hq=32, Hkv=8, D=128, P=32, lens=lens, dt="bf16",
                            num_pages=1200, max_blocks_per_seq=128, seed=seed)
        p = _params(inp, meta)
        S, _ = ops.decode_plan(p)
        assert S > 1, "the case must use split partials (scratch)"
        d = ops.device_inputs(inp, "bf16")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = ops.decode_noalloc(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                 d["context_lens"], dev_status=status)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        want = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"])
        same = _split_pair(p, d, S)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = oracle.attention(inp, **meta)
        assert_within(got, ref, tol, f"noalloc vs oracle, lens={lens}")
        assert_within(got, want.cpu().numpy().astype(np.float64), tol,
                      f"noalloc vs decode, lens={lens}")
        assert bitwise_equal(got, same.cpu().numpy()), f"noalloc vs partial + combine, lens={lens}"


def test_noalloc_rejects_partials_beyond_the_scratch():
    inp, meta = problem(B=2, Hq=16, Hkv=1, D=128, P=32, lens=(64, 64), dt="bf16", num_pages=4,
                        seed=13)
    # 64 sequences' worth of partials at 4096 splits cannot fit in 8 MiB
    p = ops.make_params(num_seqs=64, num_q_heads=16, num_kv_heads=1, head_dim=128, page_size=32,
                        num_pages=4, max_blocks_per_seq=4096, max_context_len=4096 * 32,
                        dtype="bf16", num_splits=4096)
    d = ops.device_inputs(inp, "bf16")
    with pytest.raises(ops.PaError) as e:
        ops.decode_noalloc(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["context_lens"])
    assert e.value.code == 5


def test_noalloc_single_split_plan():
    """Short contexts plan a single split; the scratch still holds it."""
    inp, meta = problem(B=4, Hq=16, Hkv=4, D=128, P=32, lens=(1, 17, 30, 32), dt="f16",
                        num_pages=12, seed=17)
    p = _params(inp, meta)
    assert ops.decode_plan(p)[0] == 1
    d = ops.device_inputs(inp, "f16")
    got = ops.decode_noalloc(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"])
    want = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert_within(got, oracle.attention(inp, **meta), workloads.TOL_16, "noalloc single split vs oracle")
    assert_within(got, want.cpu().numpy().astype(np.float64), workloads.TOL_16,
                  "noalloc single split")


def test_noalloc_host_checks_come_first():
    """Errors the host can see return before anything is enqueued: a NULL or
    misaligned out, and the options the fixed split plan does not take, even
    when the partials would also be too large for the scratch."""
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=128, P=32, lens=(64, 64), dt="bf16", num_pages=4,
                        seed=19)
    d = ops.device_inputs(inp, "bf16")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"])
    p = _params(inp, meta)
    lib = ops.load()
    fn = lib.pa_decode_noalloc
    import ctypes
    assert fn(ctypes.byref(p), *[ops._ptr(t) for t in args], None, None, None) == 1  # NULL out
    out = torch.empty(2 * 16 * 128 + 4, dtype=torch.float32, device="cuda")
    bad = ctypes.c_void_p(out.data_ptr() + 4)
    assert fn(ctypes.byref(p), *[ops._ptr(t) for t in args], bad, None, None) == 4  # misaligned
    big = dict(num_seqs=64, num_q_heads=16, num_kv_heads=2, head_dim=128, page_size=32, num_pages=4,
               max_blocks_per_seq=4096, max_context_len=4096 * 32, dtype="bf16", num_splits=4096)
    for extra in (dict(decode_q_rows=2), dict(sliding_window=8)):
        q = ops.make_params(**big)
        for k, v in extra.items():
            setattr(q, k, v)
        with pytest.raises(ops.PaError) as e:
            ops.decode_noalloc(q, *args)
        assert e.value.code == 6, extra
    q = ops.make_params(**dict(big, head_dim=256))
    with pytest.raises(ops.PaError) as e:
        ops.decode_noalloc(q, *args)
    assert e.value.code == 6
