"""Bounded device waits: a wait that runs out sets PA_DEV_TIMEOUT, the kernel
returns, and the context stays usable.

The failure is made without a fault and without a copy in flight:
pa_params.debug_timeout = 1 makes the split-KV decode kernel's warps, and the
tensor-core prefill CTA, first wait with no time allowed on a barrier that no
copy ever targets, before they issue any copy.  The kernels then take their
real timeout path (no compute, results void, unit counters still left at
zero), and the next normal call on the same buffers is correct.
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
from helpers import problem, assert_within

pytestmark = pytest.mark.gpu
TOL = workloads.TOL_16
THREADS = max(1, min(16, os.cpu_count() or 1))


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
                scale=meta["scale"], dtype=meta["q_dtype"], kv_dtype=meta["kv_dtype"])
    args.update(kw)
    return ops.make_params(**args)


@pytest.mark.parametrize("form", [0, 1, 2])
def test_decode_timeout_then_a_normal_call(form):
    lens = (1, 31, 33, 700, 2500, 90)
    inp, meta = problem(B=6, Hq=32, Hkv=8, D=128, P=32, lens=lens, dt="bf16", num_pages=120, seed=5)
    d = ops.device_inputs(inp, "bf16")
    ws = torch.zeros(ops.decode_workspace_size(_params(inp, meta)), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = _params(inp, meta, decode_form=form, debug_timeout=1)
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ops.PA_DEV_TIMEOUT
    assert torch.isfinite(out).all()
    assert int(torch.count_nonzero(ws[:4096]).item()) == 0  # counters left at zero
    status.zero_()
    p = _params(inp, meta, decode_form=form)
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_within(out.cpu().numpy(), oracle.attention(inp, threads=THREADS, **meta), TOL, "after a timeout")


def test_prefill_timeout_then_a_normal_call():
    inp, meta = problem(B=2, Hq=16, Hkv=2, D=128, P=32, lens=(300, 77), qlens=(150, 13), dt="bf16",
                        num_pages=16, seed=6)
    d = ops.device_inputs(inp, "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    total_q, max_q = int(inp["cu_q_lens"][-1]), int(np.diff(inp["cu_q_lens"]).max())
    for dbg in (1, 0):
        status.zero_()
        p = _params(inp, meta, debug_timeout=dbg)
        out = ops.prefill_chunk(p, d["q"], d["cu_q_lens"], total_q, max_q, d["k_cache"], d["v_cache"],
                                d["block_tables"], d["context_lens"], dev_status=status)
        torch.cuda.synchronize()
        if dbg:
            assert int(status.item()) == ops.PA_DEV_TIMEOUT
    assert int(status.item()) == 0
    assert_within(out.cpu().numpy(), oracle.attention(inp, threads=THREADS, **meta), TOL, "after a timeout")
