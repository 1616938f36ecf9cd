"""head_dim 256 decode (the pages' d256 decode variant: vllm.cpp PR #383,
its GQA-fused d256 kernel) against the fp64 oracle, through the C ABI."""
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

TOL = {"f16": workloads.TOL_16, "bf16": workloads.TOL_16}
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def run(inp, meta, **kw):
    bt = inp["block_tables"]
    P = meta["page_size"]
    p = ops.make_params(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                        num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"], page_size=P,
                        num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                        max_context_len=bt.shape[1] * P, scale=meta["scale"], dtype=meta["q_dtype"],
                        kv_dtype=meta["kv_dtype"], **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


CASES = [
    # B, Hq, Hkv, P, lens, dtype
    (4, 16, 8, 32, (1, 31, 33, 1500), "bf16"),   # G 2
    (3, 16, 4, 16, (15, 17, 900), "f16"),        # G 4, 16-slot pages
    (2, 32, 4, 32, (64, 2500), "bf16"),          # G 8
    (2, 4, 4, 16, (100, 777), "bf16"),           # G 1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-P{c[3]}-{c[5]}")
def test_d256_decode_matches_oracle(case):
    B, Hq, Hkv, P, lens, dt = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=256, P=P, lens=lens, dt=dt,
                        num_pages=sum((L + P - 1) // P for L in lens) + 5, seed=61)
    got, status = run(inp, meta)
    assert status == 0
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL[dt], "D256")


def test_d256_rows_and_window():
    """Two query rows per sequence (4 x 2 columns) with a 200-key window."""
    inp, meta = problem(B=2, Hq=16, Hkv=4, D=256, P=32, lens=(90, 1300), qlens=(2, 2), dt="bf16",
                        num_pages=50, seed=62)
    got, status = run(inp, meta, decode_q_rows=2, sliding_window=200)
    assert status == 0
    assert_within(got, oracle.attention(inp, window=200, threads=THREADS, **meta), TOL["bf16"], "D256 T2 W200")


def test_d256_unsupported_paths_are_rejected():
    inp, meta = problem(B=1, Hq=32, Hkv=2, D=256, P=32, lens=(40,), dt="bf16", num_pages=4, seed=63)
    with pytest.raises(ops.PaError):
        run(inp, meta)                    # G 16: two column tiles are not built for D 256
    inp, meta = problem(B=1, Hq=8, Hkv=2, D=256, P=32, lens=(40,), dt="bf16", num_pages=4, seed=64)
    with pytest.raises(ops.PaError):
        run(inp, meta, num_splits=2)      # fixed split plan
    with pytest.raises(ops.PaError):
        bt = inp["block_tables"]
        p = ops.make_params(num_seqs=1, num_q_heads=8, num_kv_heads=2, head_dim=256, page_size=32,
                            num_pages=4, max_blocks_per_seq=bt.shape[1], max_context_len=bt.shape[1] * 32,
                            dtype="bf16")
        d = ops.device_inputs(inp, "bf16")
        ops.prefill_chunk(p, d["q"], d["cu_q_lens"], 1, 1, d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"])
