"""Shared test helpers: small problem builder and comparators."""
from __future__ import annotations

import math

import numpy as np

from paged_kv_gqa_02_gb300 import inputs


def problem(B=1, Hq=4, Hkv=2, D=8, P=4, lens=(7,), qlens=None, dt="f32", kv_dt=None,
            num_pages=None, shuffle=True, seed=1, scale=None, **kw):
    """Tiny paged problem: (input dict, oracle keyword metadata)."""
    kv_dt = kv_dt or dt
    qlens = tuple(qlens) if qlens is not None else (1,) * B
    inp = inputs.make_paged_inputs(num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                   page_size=P, context_lens=lens, q_lens=qlens, q_dtype=dt,
                                   kv_dtype=kv_dt, num_pages=num_pages, shuffle=shuffle,
                                   seed=seed, **kw)
    meta = dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                scale=(1.0 / math.sqrt(D)) if scale is None else scale, q_dtype=dt,
                kv_dtype=kv_dt)
    return inp, meta


def f64(inp, meta):
    """Upcast the stored tensors of a problem to float64 (q, k, v)."""
    return (inputs.as_float64(inp["q"], meta["q_dtype"]),
            inputs.as_float64(inp["k_cache"], meta["kv_dtype"]),
            inputs.as_float64(inp["v_cache"], meta["kv_dtype"]))


def dense_ref(inp, meta):
    from oracle import dense
    q, k, v = f64(inp, meta)
    return dense.attention(q, k, v, inp["block_tables"], inp["context_lens"], inp["cu_q_lens"],
                           meta["num_q_heads"], meta["num_kv_heads"], meta["page_size"],
                           meta["scale"])


def errors(got, ref, rel_floor=1e-2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    big = np.abs(ref) > rel_floor
    max_rel = float((diff[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    finite = bool(np.isfinite(got).all())
    return max_abs, max_rel, finite


def within(got, ref, tol) -> bool:
    """The acceptance test: max abs <= tol['abs'] and, when given, max rel
    <= tol['rel'] over elements with |ref| > tol['rel_floor']."""
    a, r, finite = errors(got, ref, tol.get("rel_floor", 1e-2))
    if not finite or a > tol["abs"]:
        return False
    return "rel" not in tol or r <= tol["rel"]


def assert_within(got, ref, tol, what=""):
    a, r, finite = errors(got, ref, tol.get("rel_floor", 1e-2))
    assert within(got, ref, tol), f"{what}: max_abs={a:.3e} max_rel={r:.3e} finite={finite} tol={tol}"


def bitwise_equal(a, b) -> bool:
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and a.tobytes() == b.tobytes()
