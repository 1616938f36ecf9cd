"""pa_decode_append against the fp64 oracle, through the C ABI.

The expected result is built on the host: the new token's K/V rows are
written into a copy of the cache at row L_b - 1 of each sequence (the
append), and the oracle attends over keys [0, L_b).  Before the call the
device cache holds NaN in those rows, so a kernel that attended the row its
page copy brought in, instead of the new one, produces NaN.  After the call
the whole device cache must equal the host copy bit for bit: the new rows
are in place and nothing else changed.
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
from helpers import problem, assert_within, bitwise_equal

pytestmark = pytest.mark.gpu

TOL = {"f32": workloads.TOL_F32, "f16": workloads.TOL_16, "bf16": workloads.TOL_16}
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load()


def nan_of(dtype):
    if dtype == "bf16":
        return np.uint16(0x7FC0)
    return np.array(np.nan, dtype=inputs.storage_numpy_dtype(dtype))[()]


def host_bits(t):
    """A device cache as the host storage array (bf16 as uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def append_on_host(inp, k_new, v_new, P, fill=None):
    """Copy of the problem whose caches hold the new rows at row L-1
    (optionally, a copy holding `fill` there instead)."""
    out = dict(inp)
    k, v = inp["k_cache"].copy(), inp["v_cache"].copy()
    for b, L in enumerate(inp["context_lens"]):
        pg, slot = inp["block_tables"][b, (L - 1) // P], (L - 1) % P
        k[pg, slot] = k_new[b] if fill is None else fill
        v[pg, slot] = v_new[b] if fill is None else fill
    out["k_cache"], out["v_cache"] = k, v
    return out


def run_append(inp, meta, **kw):
    B, Hkv, D, P = len(inp["context_lens"]), meta["num_kv_heads"], meta["head_dim"], meta["page_size"]
    dt = meta["kv_dtype"]
    k_new, v_new = inputs.make_append_rows(num_seqs=B, num_kv_heads=Hkv, head_dim=D, kv_dtype=dt, seed=5)
    poisoned = append_on_host(inp, k_new, v_new, P, fill=nan_of(dt))
    expect = append_on_host(inp, k_new, v_new, P)
    bt = inp["block_tables"]
    p = ops.make_params(num_seqs=B, num_q_heads=meta["num_q_heads"], num_kv_heads=Hkv, head_dim=D,
                        page_size=P, num_pages=int(inp["num_pages"]), max_blocks_per_seq=bt.shape[1],
                        max_context_len=bt.shape[1] * P, scale=meta["scale"], dtype=meta["q_dtype"],
                        kv_dtype=dt, **kw)
    d = ops.device_inputs(poisoned, dt)
    kn, vn = ops.to_device(k_new, dt), ops.to_device(v_new, dt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ops.decode_append(p, d["q"], kn, vn, d["k_cache"], d["v_cache"], d["block_tables"],
                            d["context_lens"], dev_status=status)
    torch.cuda.synchronize()
    ref = oracle.attention(expect, threads=THREADS, **meta)
    k_after, v_after = host_bits(d["k_cache"]), host_bits(d["v_cache"])
    return out.cpu().numpy(), ref, int(status.item()), (k_after, v_after), expect


CASES = [
    # B, Hq, Hkv, D, P, lens, dtype, extra params
    (4, 16, 4, 128, 32, (1, 31, 33, 700), "bf16", {}),           # fused: 16-bit, automatic splits
    (2, 28, 4, 128, 16, (17, 300), "f16", {}),                   # fused, G = 7, 16-slot pages
    (2, 32, 2, 64, 32, (64, 129), "bf16", {}),                   # fused, G = 16 (two column tiles)
    (3, 40, 8, 128, 32, (2, 95, 1500), "f16", {}),               # fused, CTA merge and warp pieces
    (2, 12, 3, 64, 16, (16, 100), "f32", {}),                    # scatter kernel, then the fp32 path
    (3, 20, 4, 128, 32, (1, 500, 2047), "bf16", {"num_splits": 3}),  # scatter, fixed split plan
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1]}x{c[2]}-D{c[3]}-P{c[4]}-{c[6]}"
                         + ("-split" if c[7] else ""))
def test_decode_append_matches_oracle(case):
    B, Hq, Hkv, D, P, lens, dt, extra = case
    inp, meta = problem(B=B, Hq=Hq, Hkv=Hkv, D=D, P=P, lens=lens, dt=dt,
                        num_pages=sum((L + P - 1) // P for L in lens) + 9, seed=21)
    got, ref, status, (k_after, v_after), expect = run_append(inp, meta, **extra)
    assert status == 0
    assert_within(got, ref, TOL[dt], "decode_append")
    assert bitwise_equal(k_after, expect["k_cache"]), "K cache differs from the appended host copy"
    assert bitwise_equal(v_after, expect["v_cache"]), "V cache differs from the appended host copy"


def test_decode_append_full_size_14b_shape():
    """The 14B-shaped decode (40 q / 8 kv heads, D128, context 3254, P32,
    f16, shuffled 4096-page pool) with the last token appended."""
    wl = workloads.BY_NAME["decode_40x8_d128_L3254"]
    inp = wl.make_inputs()
    meta = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                page_size=wl.page_size, scale=wl.scale, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
    got, ref, status, (k_after, v_after), expect = run_append(inp, meta)
    assert status == 0
    assert_within(got, ref, TOL[wl.kv_dtype], "decode_append 14B shape")
    assert bitwise_equal(k_after, expect["k_cache"]) and bitwise_equal(v_after, expect["v_cache"])
