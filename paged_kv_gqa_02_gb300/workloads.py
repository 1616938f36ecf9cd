"""The five synthetic workloads, by shape only (no attention arithmetic).

Shapes follow the pages' own workloads:

* ``decode_12x3_d64_L1024``: crucible's 12 q / 3 kv head, head_dim 64,
  16-token page geometry at a 1024-token context (crucible paged attention
  results: the traffic paragraph and the prefill attention microbenchmark),
  fp32 Q/K/V, identity block table.
* ``decode_28x4_d128_L1641`` / ``decode_40x8_d128_L3254``: the 7B and 14B
  decode shapes of minfer docs 71/75 (byte ledger; nsys split+combine table),
  paged here with vllm.cpp's 32-token page (PR #383 numerics table), f16.
* ``ragged_b16_32x8_d128``: a 16-request continuous-batching decode batch
  (crucible README, "Paged KV cache and continuous batching"), lengths
  1/31/32/33 forced around the page boundary plus 12 seeded draws in
  [1, 4096], bf16.
* ``prefill_8x2048p512_64x8_d128``: chunked causal prefill, 8 sequences of
  2048 cached tokens plus a 512-row chunk (crucible README, "Prefill
  scheduling": row r of a chunk sees 0..=done+r), gqa 8, bf16.

Pools of 4096 pages are shuffled; sequences take disjoint pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import inputs


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "decode" or "prefill"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    q_dtype: str
    kv_dtype: str
    context_lens: tuple
    q_lens: tuple
    num_pages: int
    max_blocks_per_seq: int
    shuffle: bool
    scale: float
    seed: int = inputs.DEFAULT_SEED
    tol: dict = field(default_factory=dict)

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def total_q(self) -> int:
        return sum(self.q_lens)

    @property
    def max_context_len(self) -> int:
        return max(self.context_lens)

    def make_inputs(self, **kw):
        args = dict(num_seqs=self.num_seqs, num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    page_size=self.page_size, context_lens=self.context_lens,
                    q_lens=self.q_lens, q_dtype=self.q_dtype,
                    kv_dtype=self.kv_dtype, num_pages=self.num_pages,
                    max_blocks_per_seq=self.max_blocks_per_seq,
                    shuffle=self.shuffle, seed=self.seed)
        args.update(kw)
        return inputs.make_paged_inputs(**args)

    # ---- algorithmic byte / flop counts (K+V once per kv head, Q, O as f32)
    def elt(self, dtype: str) -> int:
        return 4 if dtype == "f32" else 2

    def kv_bytes(self) -> int:
        return (2 * sum(self.context_lens) * self.num_kv_heads * self.head_dim
                * self.elt(self.kv_dtype))

    def q_bytes(self) -> int:
        return self.total_q * self.num_q_heads * self.head_dim * self.elt(self.q_dtype)

    def o_bytes(self) -> int:
        return self.total_q * self.num_q_heads * self.head_dim * 4

    def algorithmic_bytes(self) -> int:
        return self.kv_bytes() + self.q_bytes() + self.o_bytes()

    def visible_keys(self) -> int:
        """Sum over query rows of the keys each row attends (causal bound)."""
        tot = 0
        for L, T in zip(self.context_lens, self.q_lens):
            start = L - T
            tot += T * start + T * (T + 1) // 2
        return tot

    def flops(self) -> int:
        """2 flops per multiply-add, QK^T and PV, over visible keys."""
        return 4 * self.visible_keys() * self.num_q_heads * self.head_dim


def _pages(L, P):
    return (L + P - 1) // P


def _decode(name, B, Hq, Hkv, D, P, dt, lens, num_pages, shuffle, max_blocks=None, tol=None):
    lens = tuple(int(x) for x in lens)
    return Workload(name=name, kind="decode", num_seqs=B, num_q_heads=Hq,
                    num_kv_heads=Hkv, head_dim=D, page_size=P, q_dtype=dt,
                    kv_dtype=dt, context_lens=lens, q_lens=(1,) * B,
                    num_pages=num_pages,
                    max_blocks_per_seq=max_blocks or max(_pages(L, P) for L in lens),
                    shuffle=shuffle, scale=1.0 / math.sqrt(D), tol=tol or {})


TOL_F32 = {"abs": 1e-5}
TOL_16 = {"abs": 2e-3, "rel": 1e-2, "rel_floor": 1e-2}

C1 = _decode("decode_12x3_d64_L1024", 1, 12, 3, 64, 16, "f32", [1024], 64, False, tol=TOL_F32)
C2 = _decode("decode_28x4_d128_L1641", 1, 28, 4, 128, 32, "f16", [1641], 4096, True, tol=TOL_16)
C3 = _decode("decode_40x8_d128_L3254", 1, 40, 8, 128, 32, "f16", [3254], 4096, True, tol=TOL_16)
C4 = _decode("ragged_b16_32x8_d128", 16, 32, 8, 128, 32, "bf16",
             inputs.ragged_lengths(inputs.DEFAULT_SEED, 12), 4096, True,
             max_blocks=4096 // 32, tol=TOL_16)
C5 = Workload(name="prefill_8x2048p512_64x8_d128", kind="prefill", num_seqs=8,
              num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=32,
              q_dtype="bf16", kv_dtype="bf16", context_lens=(2560,) * 8,
              q_lens=(512,) * 8, num_pages=4096, max_blocks_per_seq=80,
              shuffle=True, scale=1.0 / math.sqrt(128), tol=TOL_16)

ALL = (C1, C2, C3, C4, C5)

# Beyond the five: head_dim 256 decode (the pages' d256 variant) at the
# 14B-shaped context, gqa 2, 16-slot pages.
D256 = _decode("decode_16x8_d256_L3254", 1, 16, 8, 256, 16, "f16", [3254], 4096, True, tol=TOL_16)
# Packed small-chunk prefill: crucible's "16x16" shape (16 fresh requests of
# 16 rows, 12 q / 3 kv heads, D64, 16-token pages, f32; crucible paged
# attention results, the shape table), and the same packing at 32 q / 8 kv
# heads, D128, bf16 on the tensor cores.
PACK_F32 = Workload(name="prefill_16x16_12x3_d64_f32", kind="prefill", num_seqs=16, num_q_heads=12,
                    num_kv_heads=3, head_dim=64, page_size=16, q_dtype="f32", kv_dtype="f32",
                    context_lens=(16,) * 16, q_lens=(16,) * 16, num_pages=4096, max_blocks_per_seq=1,
                    shuffle=True, scale=1.0 / math.sqrt(64), tol=TOL_F32)
PACK_BF16 = Workload(name="prefill_16x16_32x8_d128_bf16", kind="prefill", num_seqs=16, num_q_heads=32,
                     num_kv_heads=8, head_dim=128, page_size=32, q_dtype="bf16", kv_dtype="bf16",
                     context_lens=(16,) * 16, q_lens=(16,) * 16, num_pages=4096, max_blocks_per_seq=1,
                     shuffle=True, scale=1.0 / math.sqrt(128), tol=TOL_16)
# Crucible's "4x256" prefill shape (4 fresh requests of 256 rows at offset 0,
# 12 q / 3 kv heads, D64, 16-token pages; crucible paged attention results,
# the shape table) in f32 on the CUDA cores, and in bf16 on the tensor cores
# at head_dim 64.
PACK4_F32 = Workload(name="prefill_4x256_12x3_d64_f32", kind="prefill", num_seqs=4, num_q_heads=12,
                     num_kv_heads=3, head_dim=64, page_size=16, q_dtype="f32", kv_dtype="f32",
                     context_lens=(256,) * 4, q_lens=(256,) * 4, num_pages=4096, max_blocks_per_seq=16,
                     shuffle=True, scale=1.0 / math.sqrt(64), tol=TOL_F32)
PACK4_BF16 = Workload(name="prefill_4x256_12x3_d64_bf16", kind="prefill", num_seqs=4, num_q_heads=12,
                      num_kv_heads=3, head_dim=64, page_size=16, q_dtype="bf16", kv_dtype="bf16",
                      context_lens=(256,) * 4, q_lens=(256,) * 4, num_pages=4096, max_blocks_per_seq=16,
                      shuffle=True, scale=1.0 / math.sqrt(64), tol=TOL_16)
EXTRA = (D256, PACK_F32, PACK_BF16, PACK4_F32, PACK4_BF16)

BY_NAME = {w.name: w for w in ALL + EXTRA}
