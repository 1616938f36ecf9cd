"""Packed prefill (several requests in one call) against the fp64 oracle at
full size: crucible's "16x16" shape (16 fresh requests of 16 rows, 12 q /
3 kv heads, D64, f32), the same packing at 32 q / 8 kv heads, D128, bf16 on
the tensor cores, and crucible's "4x256" shape (4 fresh requests of 256
rows, 12 q / 3 kv heads, D64) in f32 and in bf16 on the tensor cores."""
from __future__ import annotations

import os

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle
from paged_kv_gqa_02_gb300 import build, ops, workloads
from helpers import assert_within

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


@pytest.mark.parametrize("wl", (workloads.PACK_F32, workloads.PACK_BF16, workloads.PACK4_F32, workloads.PACK4_BF16),
                         ids=lambda w: w.name)
def test_packed_prefill_matches_oracle(wl):
    inp = wl.make_inputs()
    p = ops.params_for(wl)
    d = ops.device_inputs(inp, wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.prefill_chunk(p, d["q"], d["cu_q_lens"], wl.total_q, max(wl.q_lens), d["k_cache"],
                            d["v_cache"], d["block_tables"], d["context_lens"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_within(out.cpu().numpy(), oracle.attention(inp, wl, threads=THREADS), wl.tol, wl.name)
