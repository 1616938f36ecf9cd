// pa_prefill_tc.cu -- chunked causal prefill over the paged cache on the
// 5th-generation tensor cores (tcgen05 MMA, accumulators in tensor memory,
// operands staged by TMA).
//
// head_dim 64 or 128 (template parameter D), 16-bit Q/K/V.
//
// One CTA per (row-tile pair, kv head, sequence).  The MMA tile's 128 rows are
// the query heads of one kv head times 128/G consecutive chunk rows
// (row = token * G + head), so every K/V tile in shared memory serves all
// G heads (minfer doc 71: the GQA-batched shape; crucible results: K/V is
// shared across the q heads of one kv head).  Keys come in tiles of 128
// (4 pages of 32 or 8 of 16), each page one TMA box per 64-dim half.
// Row r of a chunk of T rows over a context of L keys sees keys 0..L-T+r
// (crucible README, "Prefill scheduling").
//
// Each CTA owns two such row tiles, A and B (consecutive chunk rows), that
// share every K/V tile: K/V reaches shared memory once per 256 query rows,
// and the two softmax warpgroups take turns with the tensor cores.
//
// Warp roles (320 threads):
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one thread
//              per MMA row (tensor-memory lane), online softmax in base 2
//              with a lazily raised running max, probabilities written back
//              over their scores as hi + lo 16-bit parts, and the epilogue
//              (O / l to global memory)
//   warp 8     TMA producer: Q once, then K and V tiles into their rings
//              (one lane per page issues that page's boxes)
//   warp 9     tensor-memory owner and MMA issuer (the whole warp, converged;
//              one lane elected to issue each MMA and commit)
//
// Tensor memory (512 columns): S/P of tile A [0,128), S/P of tile B
// [128,256), O of A [256,256+D), O of B [256+D,256+2D).  Per key tile j the MMA
// thread issues P_A(j).V_j, then S_A(j+1) = Q_A K_{j+1}^T once that P.V has
// finished reading P_A (same columns), then P_B(j).V_j and S_B(j+1): while
// one warpgroup computes its softmax, the tensor cores work for the other.
// Both operands of Q K^T are K-major in shared memory; P is read from
// tensor memory and V is MN-major in shared memory.
//
// Probabilities are split as p = hi + lo with both parts in the K/V type
// and both multiplied by V (two MMAs per 16 keys), so P carries ~16
// significant bits instead of 8 (bf16) or 11 (f16).
#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

#include <cudaTypedefs.h>

#include <type_traits>

namespace pa {

namespace {

constexpr int kBM = 128;         // MMA rows per row tile
constexpr int kBN = 128;         // keys per tile
constexpr int kKS = 3;           // K ring depth
constexpr int kVS = 2;           // V ring depth
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kHalfBytes = kBN * 128;     // one 64-dim half of a tile
constexpr uint32_t kNumBars = 1 + 2 * kKS + 2 * kVS + 2 * 3 + 2;

// Shared-memory layout for head_dim D (64 or 128): Q of tiles A and B, the
// K ring, the V ring, then the barriers.
template <int D> struct Smem {
    static constexpr uint32_t kTileBytes = kBN * D * 2;  // one K (or V, or Q) tile
    static constexpr uint32_t kQOff = 0;                 // Q of A, then Q of B
    static constexpr uint32_t kKOff = kQOff + 2 * kTileBytes;
    static constexpr uint32_t kVOff = kKOff + kKS * kTileBytes;
    static constexpr uint32_t kBarOff = kVOff + kVS * kTileBytes;
    static constexpr uint32_t kBytes = 1024 + kBarOff + kNumBars * 8 + 16;
};
constexpr uint64_t kWaitNs = 2000000000ull;     // a role gives up after 2 s on one barrier
constexpr uint32_t kSleepNs = 20000;            // longest sleep inside one try_wait
constexpr float kRescaleStep = 8.f;  // raise the running max only when it grows by > 2^8
constexpr uint32_t kNegInf = 0xff800000u;

// tensor-memory columns of tile x (0 = A, 1 = B): S/P, then O (D columns)
__device__ inline uint32_t col_s(int x) { return 128u * x; }
template <int D> __device__ inline uint32_t col_o(int x) { return 256u + uint32_t(D) * x; }

struct TcParams {
    const int32_t* cu_q_lens;
    const int32_t* context_lens;
    const int32_t* block_tables;
    float* out;
    uint32_t* dev_status;
    int32_t Hq, Hkv, G, tq, P, num_pages, max_blocks, max_q_len, total_q;
    int32_t n_pairs;  // row-tile pairs per (sequence, kv head)
    int32_t B;        // sequences
    int32_t debug_timeout;  // 1: the CTA's first wait (on a barrier no copy targets) gives up at once
    int32_t head_first;
    float scale_log2;  // > 0
};

// Bounded wait (by the global timer) that also gives up when another role
// has aborted.  Waiting threads sleep inside try_wait rather than spin.
__device__ inline bool wait_bar(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*abort_flag || globaltimer_ns() - t0 > kWaitNs) return false;
    }
}

__device__ inline void raise_abort(volatile uint32_t* abort_flag, uint32_t* dev_status) {
    *abort_flag = 1u;
    flag(dev_status, PA_DEV_TIMEOUT);
}

__device__ inline float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 values in one 64-bit register pair, and the paired fp32
// arithmetic of sm_100-family cores (one instruction for both lanes, each
// rounded as its scalar form).
__device__ inline uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ inline void f2_unpack(uint64_t v, uint32_t& lo, uint32_t& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ inline uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ inline uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ inline uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// hi/lo split of two probabilities (a packed fp32 pair, low = even key) into
// packed 16-bit pairs (low half = even key)
template <typename T> struct Pack;
template <> struct Pack<__nv_bfloat16> {
    // hi keeps the top 16 bits (truncation); lo = p - hi is exact in fp32 and
    // rounded to bf16, so hi + lo carries ~16 significant bits
    __device__ static inline void split(uint64_t p, uint32_t& hi, uint32_t& lo) {
        uint32_t ua, ub;
        f2_unpack(p, ua, ub);
        hi = __byte_perm(ua, ub, 0x7632);
        uint32_t da, db;
        f2_unpack(f2_sub(p, f2_pack(ua & 0xffff0000u, ub & 0xffff0000u)), da, db);
        const __nv_bfloat162 l = __floats2bfloat162_rn(__uint_as_float(da), __uint_as_float(db));
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
};
template <> struct Pack<__half> {
    __device__ static inline void split(uint64_t p, uint32_t& hi, uint32_t& lo) {
        uint32_t ua, ub;
        f2_unpack(p, ua, ub);
        const __half2 h = __floats2half2_rn(__uint_as_float(ua), __uint_as_float(ub));
        const float2 hf = __half22float2(h);
        uint32_t da, db;
        f2_unpack(f2_sub(p, f2_pack(__float_as_uint(hf.x), __float_as_uint(hf.y))), da, db);
        const __half2 l = __floats2half2_rn(__uint_as_float(da), __uint_as_float(db));
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
};

// Visible keys of one 32-key chunk as a bit mask: the first `nvis` keys,
// minus those in pages outside the pool.
__device__ inline uint32_t chunk_mask(int nvis, uint32_t pmask, int c, int P) {
    uint32_t m = nvis >= 32 ? 0xffffffffu : (nvis <= 0 ? 0u : ((1u << nvis) - 1u));
    if (P == 32) {
        if (!((pmask >> c) & 1u)) m = 0u;
    } else {  // 16-slot pages: two per chunk
        m &= (((pmask >> (2 * c)) & 1u) ? 0x0000ffffu : 0u) | (((pmask >> (2 * c + 1)) & 1u) ? 0xffff0000u : 0u);
    }
    return m;
}

__device__ inline void apply_mask(uint32_t (&r)[32], uint32_t m) {
#pragma unroll
    for (int k = 0; k < 32; ++k) r[k] = ((m >> k) & 1u) ? r[k] : kNegInf;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const TcParams a) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kD = D;
    constexpr int kHalves = D / 64;  // 64-dim (128-byte) halves of a row
    constexpr uint32_t kTileBytes = Smem<D>::kTileBytes;
    // The row-tile pairs of one (sequence, kv head) are consecutive CTAs, so
    // they run at the same time and read its K/V tiles through L2 from one
    // DRAM read; within a group the heaviest pairs come first.
    const int gb = blockIdx.x / a.n_pairs;
    const int g = gb % a.Hkv, b = gb / a.Hkv;
    const int pair = a.n_pairs - 1 - int(blockIdx.x % a.n_pairs);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G, P = a.P, tq = a.tq;

    // ---- rows of the two tiles and their causal ends ----------------------------
    if (!PA_IN(b, a.B, a.dev_status)) return;  // the whole CTA, before any barrier
    const int L = a.context_lens[b];
    const int row0 = a.cu_q_lens[b];
    const int Tq = a.cu_q_lens[b + 1] - row0;
    const bool bad = Tq < 0 || row0 < 0 || L < Tq || L > a.max_blocks * P || Tq > a.max_q_len;
    const int r_first = pair * 2 * tq;  // first chunk row of tile A
    const int t_rows = max(0, min(Tq, a.max_q_len));
    // rows of tile x that exist: below T (and the host bound), inside q/out
    auto rows_of = [&](int x) {
        const int r = r_first + x * tq;
        return row0 < 0 ? 0 : max(0, min(min(tq, t_rows - r), a.total_q - (row0 + r)));
    };
    const int n_rows_a = rows_of(0), n_rows_b = rows_of(1);
    const bool has_b = n_rows_b > 0;
    if (bad && pair == 0 && tid == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
    if (n_rows_a <= 0) return;
    if (bad) {  // no key is read; the rows are written as zeros
        const int n = (n_rows_a + n_rows_b) * G * (kD / 4);
        for (int i = tid; i < n; i += kThreads) {
            const int r = i / (G * (kD / 4)), rest = i % (G * (kD / 4));
            const int h = rest / (kD / 4), c = rest % (kD / 4);
            float* o = a.out + (int64_t(row0 + r_first + r) * a.Hq + g * G + h) * kD;
            if (PA_IN(row0 + r_first + r, a.total_q, a.dev_status))
                reinterpret_cast<float4*>(o)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int start = L - Tq;
    // keys [0, kend) are visible to some row of the CTA
    const int kend = start + r_first + (has_b ? tq + n_rows_b : n_rows_a);
    const int nt = (kend + kBN - 1) / kBN;
    const int npg = (kend + P - 1) / P;  // pages holding visible keys
    const int PT = kBN / P;              // pages per key tile
    const int32_t* table = a.block_tables + int64_t(b) * a.max_blocks;

    // ---- shared memory ------------------------------------------------------------
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + Smem<D>::kQOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + Smem<D>::kBarOff);
    uint64_t* q_full = bars;
    uint64_t* k_full = q_full + 1;
    uint64_t* k_empty = k_full + kKS;
    uint64_t* v_full = k_empty + kKS;
    uint64_t* v_empty = v_full + kVS;
    uint64_t* s_full = v_empty + kVS;  // [2]: S of tile x complete
    uint64_t* p_full = s_full + 2;     // [2]: P of tile x written (4 softmax warps)
    uint64_t* o_done = p_full + 2;     // [2]: one phase per P.V of tile x
    uint64_t* mma_done = o_done + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile uint32_t* abort_flag = tslot + 1;
    auto k_tile = [&](int st) { return base + Smem<D>::kKOff + st * kTileBytes; };
    auto v_tile = [&](int st) { return base + Smem<D>::kVOff + st * kTileBytes; };

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kKS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < kVS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(mma_done, 1);
        mbar_init(mma_done + 1, 1);  // never arrived on: the debug_timeout wait
        *abort_flag = 0u;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tslot;
    if (a.debug_timeout) {
        // Testing: a wait that runs out before any copy is issued (a barrier
        // nothing targets, no time allowed) aborts every role of the CTA.
        if (tid == 0 && !mbar_wait_ns(mma_done + 1, 0, 0)) raise_abort(abort_flag, a.dev_status);
        __syncthreads();
    }

    if (warp == kProducerWarp) {
        // ================================ producer ================================
        const int xc = a.head_first ? g : 0, yc = a.head_first ? 0 : g;
        const bool q_issued = !*abort_flag;
        if (lane == 0 && q_issued) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            // full box bytes count even where the box leaves the tensor (zero fill)
            const uint32_t qbytes = uint32_t(kHalves) * 128u * uint32_t(G * tq);
            mbar_arrive_expect_tx(q_full, has_b ? 2 * qbytes : qbytes);
            for (int x = 0; x < (has_b ? 2 : 1); ++x)
                for (int hh = 0; hh < kHalves; ++hh)
                    tma_load_3d(sQ + x * kTileBytes + hh * kHalfBytes, &tmQ, q_full, 64 * hh, g * G,
                                row0 + r_first + x * tq);
        }
        // lane p issues both halves of page p of each tile
        auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int pg) {
            if (lane == 0) mbar_arrive_expect_tx(bar, kTileBytes);
            __syncwarp();
            if (lane < PT)
#pragma unroll
                for (int hh = 0; hh < kHalves; ++hh)
                    tma_load_4d(dst + hh * kHalfBytes + lane * P * 128, map, bar, 64 * hh, xc, yc, pg);
        };
        int kq = 0, vq = 0;  // tiles issued
        bool ok = q_issued;
        for (int j = 0; ok && j < nt; ++j) {
            // physical page of lane's slot in tile j (out-of-pool entries flagged, read as zeros)
            int pg = a.num_pages;  // beyond the tensor: the box reads as zeros
            const int idx = j * PT + lane;
            if (lane < PT && idx < npg && PA_IN(idx, a.max_blocks, a.dev_status)) {
                const int e = table[idx];
                if (e >= 0 && e < a.num_pages)
                    pg = e;
                else
                    flag(a.dev_status, PA_DEV_BAD_PAGE);
            }
            const int sk = j % kKS, sv = j % kVS;
            if (j >= kKS) ok = __all_sync(0xffffffffu, wait_bar(&k_empty[sk], ((j / kKS) - 1) & 1, abort_flag));
            if (!ok) break;
            load_tile(k_tile(sk), &tmK, &k_full[sk], pg);
            kq = j + 1;
            if (j >= kVS) ok = __all_sync(0xffffffffu, wait_bar(&v_empty[sv], ((j / kVS) - 1) & 1, abort_flag));
            if (!ok) break;
            load_tile(v_tile(sv), &tmV, &v_full[sv], pg);
            vq = j + 1;
        }
        if (lane == 0) {
            if (!ok) raise_abort(abort_flag, a.dev_status);
            // never leave the CTA with copies in flight
            for (int j = max(0, kq - kKS); j < kq; ++j) mbar_wait_ns(&k_full[j % kKS], (j / kKS) & 1, kWaitNs);
            for (int j = max(0, vq - kVS); j < vq; ++j) mbar_wait_ns(&v_full[j % kVS], (j / kVS) & 1, kWaitNs);
            if (q_issued && !mbar_wait_ns(q_full, 0, kWaitNs)) flag(a.dev_status, PA_DEV_TIMEOUT);
        }
    } else if (warp == kMmaWarp) {
        // ================================== MMA ===================================
        // The whole warp runs this role, converged; one elected lane issues the
        // MMAs and commits (the *_elect forms).  Issue from a lone lane in a
        // divergent branch was measured at ~100 cycles an MMA once the softmax
        // warps of the same sub-partition were busy, against the 64 cycles an
        // MMA of this shape takes.
        const uint32_t idQK = tc::idesc_f16(kBM, kBN, kBf16, false);
        const uint32_t idPV = tc::idesc_f16(kBM, kD, kBf16, true);
        const int nx = has_b ? 2 : 1;
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
        };
        bool ok = wait_all(q_full, 0);
        tc::fence_after_sync();
        // descriptors: the high word is shared, low words advance by offset >> 4
        const uint32_t hi_d = tc::desc_hi_sw128(1024);
        const uint32_t q_lo = tc::desc_lo(smem_u32(sQ), 16);
        const uint32_t k_lo = tc::desc_lo(smem_u32(k_tile(0)), 16);
        const uint32_t v_lo = tc::desc_lo(smem_u32(v_tile(0)), kHalfBytes);
        // S_x = Q_x K_j^T into the columns of tile x
        auto qk = [&](int x, int j) {
            const uint32_t qx = q_lo + x * (kTileBytes >> 4);
            const uint32_t kx = k_lo + (j % kKS) * (kTileBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
                tc::mma_ss_elect(tm + col_s(x), tc::make_desc(qx + off, hi_d), tc::make_desc(kx + off, hi_d), idQK,
                                 ks > 0);
            }
            tc::commit_elect(&s_full[x]);
        };
        // O_x += P_x V_j, P_x read from the score columns of tile x
        auto pv = [&](int x, int j) {
            const uint32_t vx = v_lo + (j % kVS) * (kTileBytes >> 4);
            const uint32_t p_col = tm + col_s(x), o_col = tm + col_o<D>(x);
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks) {
                // 16 keys: 8-row core groups 1024 B apart, dim halves 16 KB apart.
                // P of keys 32c..32c+31 sits in columns 32c (hi, 16) and 32c+16 (lo, 16).
                const uint64_t bd = tc::make_desc(vx + ks * (2048 >> 4), hi_d);
                const uint32_t col = p_col + 32 * (ks >> 1) + 8 * (ks & 1);
                tc::mma_ts_elect(o_col, col, bd, idPV, j > 0 || ks > 0);
                tc::mma_ts_elect(o_col, col + 16, bd, idPV, true);
            }
            tc::commit_elect(&o_done[x]);
        };
        if (ok) ok = wait_all(&k_full[0], 0);
        if (ok) {
            tc::fence_after_sync();
            for (int x = 0; x < nx; ++x) qk(x, 0);
            tc::commit_elect(&k_empty[0]);
        }
        // per key tile and row tile x: P_x.V, then the next S_x, which
        // overwrites P_x and so waits for that P.V to finish
        for (int j = 0; ok && j < nt; ++j) {
            for (int x = 0; ok && x < nx; ++x) {
                ok = wait_all(&p_full[x], j & 1);
                if (ok && x == 0) ok = wait_all(&v_full[j % kVS], (j / kVS) & 1);
                if (!ok) break;
                tc::fence_after_sync();
                pv(x, j);
                if (x == nx - 1) tc::commit_elect(&v_empty[j % kVS]);
                if (j + 1 < nt) {
                    if (x == 0) ok = wait_all(&k_full[(j + 1) % kKS], ((j + 1) / kKS) & 1);
                    if (ok) ok = wait_all(&o_done[x], j & 1);
                    if (!ok) break;
                    tc::fence_after_sync();
                    qk(x, j + 1);
                    if (x == nx - 1) tc::commit_elect(&k_empty[(j + 1) % kKS]);
                }
            }
        }
        if (!ok && lane == 0) raise_abort(abort_flag, a.dev_status);
        // every MMA issued so far has finished before tensor memory is freed
        tc::commit_elect(mma_done);
        if (!__all_sync(0xffffffffu, mbar_wait_ns(mma_done, 0, kWaitNs)) && lane == 0)
            flag(a.dev_status, PA_DEV_TIMEOUT);
    } else if (warp < 4 || has_b) {
        // ================================= softmax =================================
        const int x = warp >> 2;  // tile
        const int quad = warp & 3;
        const int m = quad * 32 + lane;  // MMA row = tensor-memory lane
        const uint32_t lane_addr = uint32_t(quad * 32) << 16;
        const int t = m / G, h = m - (m / G) * G;
        const int n_rows = x ? n_rows_b : n_rows_a;
        const int r_tile = r_first + x * tq;
        const bool row_ok = t < tq && t < n_rows;
        const int lim = row_ok ? start + r_tile + t + 1 : 0;  // keys [0, lim)
        const float sl2 = a.scale_log2;
        const uint32_t sbase = tm + lane_addr + col_s(x);
        const uint32_t obase = tm + lane_addr + col_o<D>(x);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        // Table entry of page `lane` of key tile jj (0 for lanes past the
        // tile's pages, which counts as a page inside the pool); loaded a key
        // tile ahead of its use.
        auto entry = [&](int jj) -> int {
            const int idx = jj * PT + lane;
            return lane < PT && idx < npg && PA_IN(idx, a.max_blocks, a.dev_status) ? __ldg(table + idx) : 0;
        };
        int e_cur = entry(0);
        for (int j = 0; j < nt; ++j) {
            const int k0 = j * kBN;
            const int e_nxt = j + 1 < nt ? entry(j + 1) : 0;
            ok = __all_sync(0xffffffffu, wait_bar(&s_full[x], j & 1, abort_flag));
            if (!ok) break;
            tc::fence_after_sync();
            // pages of this tile outside the pool are skipped (flagged by the producer)
            const uint32_t pmask = __ballot_sync(0xffffffffu, e_cur >= 0 && e_cur < a.num_pages);
            e_cur = e_nxt;
            const bool full = (k0 + kBN <= lim) && pmask == 0xffffffffu;

            // ---- pass 1: row max of the raw scores (scale > 0 keeps the order),
            // 32 columns at a time.  Both passes are rolled loops: the code the
            // softmax warps run stays small, so it does not push the MMA
            // thread's code (same sub-partition) out of the instruction cache.
            float mx = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc::ld_32x32b_x32(sbase + 32 * c, r);
                tc::wait_ld();
                tc::reg_fence(r);
                if (!full) apply_mask(r, chunk_mask(lim - k0 - 32 * c, pmask, c, P));
                float m0 = mx, m1 = -INFINITY;
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    m0 = max3(m0, __uint_as_float(r[k]), __uint_as_float(r[k + 1]));
                    m1 = max3(m1, __uint_as_float(r[k + 2]), __uint_as_float(r[k + 3]));
                }
                mx = fmaxf(m0, m1);
            }
            const float mt = mx * sl2;  // -inf when nothing is visible
            const bool need = mt > m_run + kRescaleStep;
            const float alpha = need ? ex2(m_run - mt) : 1.f;
            if (need) m_run = mt;
            l_run *= alpha;

            // O_x is rescaled in place: P_x(j-1).V has finished (S_x(j) was
            // issued after it)
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
                for (int c = 0; c < kD / 16; ++c) {
                    uint32_t ro[16];
                    tc::ld_32x32b_x16(obase + 16 * c, ro);
                    tc::wait_ld();
                    tc::reg_fence(ro);
#pragma unroll
                    for (int k = 0; k < 16; ++k) ro[k] = __float_as_uint(__uint_as_float(ro[k]) * alpha);
                    tc::st_32x32b_x16(obase + 16 * c, ro);
                }
            }

            // ---- pass 2: p = 2^(s * scale_log2 - m_run), split hi + lo in place
            // (hi over the even key of a pair, lo over the odd) and written over
            // the scores: keys 32c.. -> columns 32c (hi) and 32c + 16 (lo)
            // Key pairs go through the paired fp32 instructions: the scaled
            // exponent, the two running sums (even and odd keys) and the lo
            // remainder take one instruction a pair.
            const float nmu = m_run == -INFINITY ? 0.f : -m_run;
            const uint64_t sl2_2 = f2_pack(__float_as_uint(sl2), __float_as_uint(sl2));
            const uint64_t nmu_2 = f2_pack(__float_as_uint(nmu), __float_as_uint(nmu));
            uint64_t sum_2 = f2_pack(0u, 0u);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tc::ld_32x32b_x32(sbase + 32 * c, r);
                tc::wait_ld();
                tc::reg_fence(r);
                if (!full) apply_mask(r, chunk_mask(lim - k0 - 32 * c, pmask, c, P));
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    uint32_t z0, z1;
                    f2_unpack(f2_fma(f2_pack(r[2 * w], r[2 * w + 1]), sl2_2, nmu_2), z0, z1);
                    const uint64_t pp = f2_pack(__float_as_uint(ex2(__uint_as_float(z0))),
                                                __float_as_uint(ex2(__uint_as_float(z1))));
                    sum_2 = f2_add(sum_2, pp);
                    Pack<T>::split(pp, r[2 * w], r[2 * w + 1]);
                }
                tc::st_32x32b_x16_stride2<0>(sbase + 32 * c, r);
                tc::st_32x32b_x16_stride2<1>(sbase + 32 * c + 16, r);
            }
            uint32_t sum0, sum1;
            f2_unpack(sum_2, sum0, sum1);
            l_run += __uint_as_float(sum0) + __uint_as_float(sum1);
            tc::wait_st();

            // slots past the context in its last page may hold anything (NaN):
            // tile A's warps zero those V rows (before either P.V reads them)
            const int zlo = L - k0, zhi = min(kBN, npg * P - k0);
            if (x == 0 && zlo < zhi) {
                const int sv = j % kVS;
                ok = __all_sync(0xffffffffu, wait_bar(&v_full[sv], (j / kVS) & 1, abort_flag));
                if (!ok) break;
                uint8_t* sV = v_tile(sv);
                for (int i = m; i < (zhi - zlo) * (kD / 8); i += kBM) {
                    const int row = zlo + i / (kD / 8), c = i % (kD / 8);
                    *reinterpret_cast<uint4*>(sV + (c >> 3) * kHalfBytes + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
        }

        // ---- epilogue: O / l ------------------------------------------------------
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(&o_done[x], (nt - 1) & 1, abort_flag));
        if (ok) {
            tc::fence_after_sync();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            float* orow = a.out + (int64_t(row0 + r_tile + t) * a.Hq + g * G + h) * kD;
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t ra[32];
                tc::ld_32x32b_x32(obase + 32 * c, ra);
                tc::wait_ld();
                tc::reg_fence(ra);
                if (row_ok && PA_IN(row0 + r_tile + t, a.total_q, a.dev_status)) {
                    float4* dst = reinterpret_cast<float4*>(orow + 32 * c);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(ra[4 * k]) * inv, __uint_as_float(ra[4 * k + 1]) * inv,
                                             __uint_as_float(ra[4 * k + 2]) * inv,
                                             __uint_as_float(ra[4 * k + 3]) * inv);
                }
            }
        } else {
            raise_abort(abort_flag, a.dev_status);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tm, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <typename T, int D>
cudaError_t launch_typed(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const TcParams& p,
                         int n_ctas, cudaStream_t st) {
    auto kern = prefill_tc<T, D>;
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Smem<D>::kBytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<dim3(n_ctas), kThreads, Smem<D>::kBytes, st>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(pa_dtype dt, int D, int P, int G, float scale) {
    return dt != PA_F32 && (D == 64 || D == 128) && (P == 16 || P == 32) && G >= 1 && G <= kMaxGroup &&
           scale > 0.f;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st) {
    if (!prefill_tc_supported(dt, D, P, a.group, a.scale_log2)) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int G = a.group;
    const int tq = kBM / G;
    const CUtensorMapDataType tdt =
        dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // Q as (head_dim, q head, row); box: 64 dims x G heads x tq rows
    CUtensorMap mq, mk, mv;
    {
        cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(a.num_q_heads), cuuint64_t(a.total_q)};
        cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(a.num_q_heads) * D * 2};
        cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(tq)};
        cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&mq, tdt, 3, const_cast<void*>(a.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // K/V pool as (head_dim, kv head, slot, page) with the middle two in
    // stride order; the box is one page of one kv head, 64 dims at a time
    const int head_first = a.head_stride <= a.token_stride;
    {
        cuuint64_t dims[4], strides[3];
        cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
        dims[0] = D;
        dims[3] = cuuint64_t(a.num_pages);
        strides[2] = cuuint64_t(a.page_stride) * 2;
        if (head_first) {
            dims[1] = a.num_kv_heads;
            dims[2] = P;
            strides[0] = cuuint64_t(a.head_stride) * 2;
            strides[1] = cuuint64_t(a.token_stride) * 2;
            box[0] = 64; box[1] = 1; box[2] = P; box[3] = 1;
        } else {
            dims[1] = P;
            dims[2] = a.num_kv_heads;
            strides[0] = cuuint64_t(a.token_stride) * 2;
            strides[1] = cuuint64_t(a.head_stride) * 2;
            box[0] = 64; box[1] = P; box[2] = 1; box[3] = 1;
        }
        if (enc(&mk, tdt, 4, const_cast<void*>(a.k), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (enc(&mv, tdt, 4, const_cast<void*>(a.v), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    TcParams p;
    p.cu_q_lens = a.cu_q_lens;
    p.context_lens = a.context_lens;
    p.block_tables = a.block_tables;
    p.out = a.out;
    p.dev_status = a.dev_status;
    p.Hq = a.num_q_heads;
    p.Hkv = a.num_kv_heads;
    p.G = G;
    p.tq = tq;
    p.P = P;
    p.num_pages = a.num_pages;
    p.max_blocks = a.max_blocks_per_seq;
    p.max_q_len = a.max_q_len;
    p.total_q = a.total_q;
    p.B = a.num_seqs;
    p.debug_timeout = a.debug_timeout;
    p.head_first = head_first;
    p.scale_log2 = a.scale_log2;
    const int64_t n_pairs = (a.max_q_len + 2 * tq - 1) / (2 * tq);  // pairs of row tiles
    const int64_t n_ctas = n_pairs * a.num_kv_heads * a.num_seqs;
    if (n_ctas > 0x7fffffff) return cudaErrorInvalidValue;
    p.n_pairs = int32_t(n_pairs);
    if (D == 64)
        return dt == PA_BF16 ? launch_typed<__nv_bfloat16, 64>(mq, mk, mv, p, int(n_ctas), st)
                             : launch_typed<__half, 64>(mq, mk, mv, p, int(n_ctas), st);
    return dt == PA_BF16 ? launch_typed<__nv_bfloat16, 128>(mq, mk, mv, p, int(n_ctas), st)
                         : launch_typed<__half, 128>(mq, mk, mv, p, int(n_ctas), st);
}

}  // namespace pa
