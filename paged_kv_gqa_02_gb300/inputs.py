"""Seeded synthetic inputs for paged grouped-query attention.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It holds none of the attention arithmetic: it only draws numbers and
lays them out (paged pools, block tables, lengths).

Recipe (counter-based, so any element can be drawn on its own):

* ``splitmix64``: the published mixer of Steele, Lea and Flood (2014),
  output ``n`` (0-based) of a stream seeded ``s`` is ``mix(s + (n+1)*gamma)``
  with ``gamma = 0x9E3779B97F4A7C15``.
* Each tensor has its own stream: ``seed ^ (tensor_id * gamma mod 2**64)``.
* N(0,1) samples come from the Box-Muller transform in double precision:
  element ``i`` uses the uniform pair ``(2*(i//2), 2*(i//2)+1)``;
  ``u1 = ((x >> 11) + 1) * 2**-53`` lies in (0, 1], ``u2 = (x >> 11) * 2**-53``;
  even ``i`` takes ``r*cos(2*pi*u2)``, odd ``i`` takes ``r*sin(2*pi*u2)``.
* Rounding to the storage dtype is round-to-nearest-even: double -> f32,
  double -> f16 directly, and double -> f32 -> bf16 for bf16.
* The default seed is 20260908, the tensor seed of the crucible paged
  attention results page (the paragraph on the final tensor run).

bf16 tensors are returned as ``uint16`` bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1
DEFAULT_SEED = 20260908

# tensor ids of the per-tensor streams
TID_Q = 1
TID_K = 2
TID_V = 3
TID_TABLE = 4
TID_K_NEW = 6   # new-token K rows of a decode-with-append call
TID_V_NEW = 7

DTYPES = ("f32", "f16", "bf16")


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def splitmix64_at(seed: int, idx: np.ndarray) -> np.ndarray:
    """Outputs number ``idx`` (0-based, uint64 array) of the stream ``seed``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + (idx + np.uint64(1)) * np.uint64(GAMMA)
        return _mix(z)


class SplitMix64:
    """Sequential splitmix64 stream (used for lengths and shuffles)."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + GAMMA) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)


def stream_seed(seed: int, tensor_id: int) -> int:
    return (seed ^ ((tensor_id * GAMMA) & MASK64)) & MASK64


def normal_at(seed: int, idx: np.ndarray) -> np.ndarray:
    """N(0,1) doubles for element indices ``idx`` of the stream ``seed``."""
    idx = np.asarray(idx, dtype=np.uint64)
    pair = idx >> np.uint64(1)
    x1 = splitmix64_at(seed, pair * np.uint64(2))
    x2 = splitmix64_at(seed, pair * np.uint64(2) + np.uint64(1))
    u1 = ((x1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (x2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    odd = (idx & np.uint64(1)).astype(bool)
    return np.where(odd, r * np.sin(th), r * np.cos(th))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even f32 -> bf16, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round doubles to the storage dtype (bf16 -> uint16 bits)."""
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype}")


def as_float64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact upcast of a stored tensor to double (bf16 given as bits)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def normal_tensor(seed: int, tensor_id: int, shape, dtype: str,
                  flat_index: np.ndarray | None = None) -> np.ndarray:
    s = stream_seed(seed, tensor_id)
    n = int(np.prod(shape))
    idx = np.arange(n, dtype=np.uint64) if flat_index is None else flat_index
    return round_to(normal_at(s, idx), dtype).reshape(shape)


def fisher_yates(n: int, seed: int) -> np.ndarray:
    """Permutation of 0..n-1: for i = n-1 .. 1, swap i with next() % (i+1)."""
    g = SplitMix64(seed)
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = g.next() % (i + 1)
        p[i], p[j] = p[j], p[i]
    return p


def ragged_lengths(seed: int, n_random: int, forced=(1, 31, 32, 33), max_len: int = 4096):
    """``forced`` lengths, then ``n_random`` draws of ``1 + next() % max_len``."""
    g = SplitMix64(seed)
    out = list(forced)
    for _ in range(n_random):
        out.append(1 + g.next() % max_len)
    return out


def storage_numpy_dtype(dtype: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]


def make_paged_inputs(*, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                      head_dim: int, page_size: int, context_lens, q_lens,
                      q_dtype: str, kv_dtype: str, num_pages: int | None = None,
                      max_blocks_per_seq: int | None = None, shuffle: bool = True,
                      seed: int = DEFAULT_SEED, unused_fill: float = 0.0,
                      unused_table_entry: int = -1):
    """Build one paged-attention problem.

    Layouts (all C-contiguous):
      q            [total_q][Hq][D]           (rows of seq s are cu_q_lens[s]..)
      k_cache      [num_pages][P][Hkv][D]     (same for v_cache)
      block_tables [B][max_blocks_per_seq] int32, entries past ceil(L/P) are
                   ``unused_table_entry``
      context_lens [B] int32 (history + this call's query rows)
      cu_q_lens    [B+1] int32

    Physical pages come from a Fisher-Yates shuffle of the pool (or the
    identity when ``shuffle`` is False); sequence s takes the next
    ceil(L_s/P) pages of that order, so no two sequences share a page.
    Only referenced pages are drawn; the rest hold ``unused_fill``.
    """
    B, Hq, Hkv, D, P = num_seqs, num_q_heads, num_kv_heads, head_dim, page_size
    context_lens = [int(x) for x in context_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(context_lens) == B and len(q_lens) == B
    n_blocks = [(L + P - 1) // P for L in context_lens]
    need = sum(n_blocks)
    if num_pages is None:
        num_pages = max(need, 1)
    assert need <= num_pages, "pool too small"
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(max(n_blocks), 1)
    order = (fisher_yates(num_pages, stream_seed(seed, TID_TABLE)) if shuffle
             else np.arange(num_pages, dtype=np.int64))
    bt = np.full((B, max_blocks_per_seq), unused_table_entry, dtype=np.int32)
    pos = 0
    for s in range(B):
        bt[s, :n_blocks[s]] = order[pos:pos + n_blocks[s]]
        pos += n_blocks[s]
    used = np.sort(order[:need])

    page_elems = P * Hkv * D
    kv_np = storage_numpy_dtype(kv_dtype)
    fill = round_to(np.array([unused_fill], dtype=np.float64), kv_dtype)[0]
    k = np.full((num_pages, P, Hkv, D), fill, dtype=kv_np)
    v = np.full((num_pages, P, Hkv, D), fill, dtype=kv_np)
    if need:
        flat = (used.astype(np.uint64)[:, None] * np.uint64(page_elems)
                + np.arange(page_elems, dtype=np.uint64)[None, :]).reshape(-1)
        k[used] = normal_tensor(seed, TID_K, (need, P, Hkv, D), kv_dtype, flat)
        v[used] = normal_tensor(seed, TID_V, (need, P, Hkv, D), kv_dtype, flat)
    total_q = sum(q_lens)
    q = normal_tensor(seed, TID_Q, (total_q, Hq, D), q_dtype)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return dict(q=q, k_cache=k, v_cache=v, block_tables=bt,
                context_lens=np.asarray(context_lens, dtype=np.int32),
                cu_q_lens=cu, num_pages=num_pages,
                max_blocks_per_seq=max_blocks_per_seq)


def make_append_rows(*, num_seqs: int, num_kv_heads: int, head_dim: int, kv_dtype: str,
                     seed: int = DEFAULT_SEED):
    """The new token's K and V rows of a decode-with-append call:
    two [B][Hkv][D] arrays, N(0,1) rounded to the storage dtype."""
    shape = (num_seqs, num_kv_heads, head_dim)
    return (normal_tensor(seed, TID_K_NEW, shape, kv_dtype),
            normal_tensor(seed, TID_V_NEW, shape, kv_dtype))
