"""The K/V pool in head-major order ([page][kv head][slot][dim], passed
through pa_params' page / token / head strides) gives the same output bits
as the default slot-major order ([page][slot][kv head][dim]) on every
kernel: the 16-bit split-KV decode (both forms), the fp32 decode, the
tensor-core prefill at head_dim 64 and 128, and the fp32 prefill.  The
kernels address pages through the strides alone, so moving the storage must
not move the arithmetic."""
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

THREADS = max(1, min(16, os.cpu_count() or 1))
TOL = {"f32": workloads.TOL_F32, "f16": workloads.TOL_16, "bf16": workloads.TOL_16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def head_major(inp):
    """The same pool with each page's kv heads outermost, and its strides."""
    k, v = inp["k_cache"], inp["v_cache"]
    n, P, H, D = k.shape
    moved = dict(inp, k_cache=np.ascontiguousarray(k.transpose(0, 2, 1, 3)),
                 v_cache=np.ascontiguousarray(v.transpose(0, 2, 1, 3)))
    return moved, (H * P * D, D, P * D)  # page, token (slot), head strides in elements


def run(inp, meta, prefill, strides=(0, 0, 0), **kw):
    bt = inp["block_tables"]
    P = meta["page_size"]
    p = ops.make_params(num_seqs=len(inp["context_lens"]), num_q_heads=meta["num_q_heads"],
                        num_kv_heads=meta["num_kv_heads"], head_dim=meta["head_dim"], page_size=P,
                        num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                        max_context_len=bt.shape[1] * P, scale=meta["scale"], dtype=meta["q_dtype"],
                        kv_dtype=meta["kv_dtype"], strides=strides, **kw)
    d = ops.device_inputs(inp, meta["kv_dtype"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if prefill:
        qlens = np.diff(inp["cu_q_lens"])
        out = ops.prefill_chunk(p, d["q"], d["cu_q_lens"], int(inp["cu_q_lens"][-1]), int(qlens.max()),
                                d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                dev_status=status)
    else:
        out = ops.decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                         dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(status.item())


CASES = [
    # name, prefill, B, Hq, Hkv, D, P, lens, qlens, dtype, extra params
    ("decode-v1-pair", False, 4, 32, 8, 128, 32, (1, 33, 700, 2000), None, "bf16", {}),
    ("decode-v1-counted", False, 3, 16, 4, 128, 16, (5, 900, 64), None, "f16",
     {"decode_form": ops.PA_FORM_COUNTED}),
    ("decode-v1-d64", False, 2, 16, 2, 64, 32, (300, 31), None, "bf16", {}),
    ("decode-f32", False, 2, 12, 3, 64, 16, (1024, 17), None, "f32", {}),
    ("prefill-tc-d128", True, 2, 32, 8, 128, 32, (300, 129), (100, 129), "bf16", {}),
    ("prefill-tc-d64", True, 2, 12, 3, 64, 16, (257, 64), (64, 64), "f16", {}),
    ("prefill-f32", True, 2, 16, 4, 64, 32, (400, 100), (150, 100), "f32", {}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_head_major_pool_matches_slot_major(case):
    name, prefill, B, Hq, Hkv, D, P, lens, qlens, dt, kw = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, qlens=qlens, dt=dt,
                        num_pages=sum((L + P - 1) // P for L in lens) + 5, seed=len(name) * 7 + B)
    base, s0 = run(inp, meta, prefill, **kw)
    moved, strides = head_major(inp)
    got, s1 = run(moved, meta, prefill, strides=strides, **kw)
    assert s0 == 0 and s1 == 0
    assert bitwise_equal(got, base), name
    assert_within(got, oracle.attention(inp, threads=THREADS, **meta), TOL[dt], name)
