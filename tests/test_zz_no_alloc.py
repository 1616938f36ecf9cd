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

from paged_kv_gqa_02_gb300 import build, ops, workloads
from helpers import problem, assert_within

pytestmark = pytest.mark.gpu


def _params(inp, meta, **kw):
    bt = inp["block_tables"]
    return ops.make_params(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                           num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"],
                           page_size=meta["page_size"], num_pages=int(inp["num_pages"]),
                           max_blocks_per_seq=bt.shape[1],
                           max_context_len=bt.shape[1] * meta["page_size"], scale=meta["scale"],
                           dtype=meta["q_dtype"], kv_dtype=meta["kv_dtype"], **kw)


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    """Two consecutive calls with different batches: each equals pa_decode
    (with a caller workspace) within the decode test tolerance, so the
    scratch left by the first call does not leak into the second."""
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
        want = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"])
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_within(got.cpu().numpy(), want.cpu().numpy().astype(np.float64), tol,
                      f"noalloc vs decode, lens={lens}")


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
    assert_within(got.cpu().numpy(), want.cpu().numpy().astype(np.float64), workloads.TOL_16,
                  "noalloc single split")
