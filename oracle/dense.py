"""Second, independently written oracle path: dense materialisation.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  Used only to pin the C
oracle on tiny shapes.  It differs from it on purpose in every step that
could hide a mistake:

* it first builds a dense ``[L][Hkv][D]`` copy of each sequence's K and V by
  walking logical positions and reading ``block_tables`` (the pool layout of
  the crucible README, "Layout, and why it was nearly free"), instead of
  translating inside the score loop;
* it expands kv heads to q heads with ``np.repeat`` (the repeat_interleave
  form of the GQA mapping, crucible README test list), instead of an index
  division;
* it applies the causal bound as a boolean mask over a full score matrix
  (crucible README, "Prefill scheduling": row r sees 0 ..= done + r);
* softmax and the weighted sum are numpy matrix operations in float64.

All arguments are float64 arrays already upcast from storage.
"""
from __future__ import annotations

import numpy as np


def gather_dense(pool: np.ndarray, table_row: np.ndarray, L: int, page_size: int) -> np.ndarray:
    """pool [num_pages][P][Hkv][D] -> dense [L][Hkv][D] for one sequence."""
    out = np.empty((L,) + pool.shape[2:], dtype=pool.dtype)
    for j in range(L):
        page = int(table_row[j // page_size])
        if not 0 <= page < pool.shape[0]:
            raise IndexError(f"page {page} outside the pool")
        out[j] = pool[page, j % page_size]
    return out


def attention(q, k_pool, v_pool, block_tables, context_lens, cu_q_lens,
              num_q_heads, num_kv_heads, page_size, scale, window=0):
    """q [total_q][Hq][D] (float64) -> out [total_q][Hq][D] (float64)."""
    group = num_q_heads // num_kv_heads
    out = np.zeros_like(q, dtype=np.float64)
    for s in range(len(context_lens)):
        L = int(context_lens[s])
        r0, r1 = int(cu_q_lens[s]), int(cu_q_lens[s + 1])
        T = r1 - r0
        if T == 0:
            continue
        K = np.repeat(gather_dense(k_pool, block_tables[s], L, page_size), group, axis=1)
        V = np.repeat(gather_dense(v_pool, block_tables[s], L, page_size), group, axis=1)
        Q = q[r0:r1]                                   # [T][Hq][D]
        S = np.einsum("thd,jhd->htj", Q, K) * scale     # [Hq][T][L]
        pos = (L - T) + np.arange(T)                    # absolute row positions
        visible = np.arange(L)[None, :] <= pos[:, None]  # [T][L]
        if window > 0:                                  # only the last `window` keys of each row
            visible &= np.arange(L)[None, :] > pos[:, None] - window
        S = np.where(visible[None], S, -np.inf)
        S = S - S.max(axis=2, keepdims=True)
        W = np.exp(S)
        W = W / W.sum(axis=2, keepdims=True)
        out[r0:r1] = np.einsum("htj,jhd->thd", W, V)
    return out
