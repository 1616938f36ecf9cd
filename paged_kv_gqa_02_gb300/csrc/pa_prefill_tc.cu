// pa_prefill_tc.cu -- chunked causal prefill over the paged cache on the
// 5th-generation tensor cores (tcgen05 MMA, accumulators in tensor memory,
// operands staged by TMA).
//
// One CTA per (row tile, kv head, sequence).  The MMA tile's 128 rows are
// the query heads of one kv head times 128/G consecutive chunk rows
// (row = token * G + head), so every K/V tile in shared memory serves all
// G heads (minfer doc 71: the GQA-batched shape; crucible results: K/V is
// shared across the q heads of one kv head).  Keys come in tiles of 128
// (4 pages of 32 or 8 of 16), each page one TMA box per 64-dim half.
// Row r of a chunk of T rows over a context of L keys sees keys 0..L-T+r
// (crucible README, "Prefill scheduling").
//
// Warp roles (192 threads):
//   warp 0     TMA producer: Q once, then K/V tiles into a 3-stage ring
//   warp 1     tensor-memory owner and MMA issuer (one thread)
//   warps 2-5  softmax: one thread per MMA row (tensor-memory lane), online
//              softmax in base 2 with a lazily raised running max, the
//              probabilities written back to tensor memory as hi + lo
//              16-bit parts, and the epilogue (O / l to global memory)
//
// Tensor memory (512 columns): S double buffer [0,256), P hi [256,320),
// P lo [320,384), O [384,512).  Per key tile j the MMA thread issues
// S_j = Q K_j^T (both operands K-major from shared memory), then, once the
// softmax has written P_{j-1}, O += P_{j-1} V_{j-1} (P from tensor memory,
// V MN-major from shared memory).
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

constexpr int kD = 128;          // head_dim served by this kernel
constexpr int kBM = 128;         // MMA rows
constexpr int kBN = 128;         // keys per tile
constexpr int kStages = 3;       // K/V ring depth
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kBN * kD * 2;  // one K (or V) tile
constexpr uint32_t kHalfBytes = kBN * 128;     // one 64-dim half of a tile
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kQOff = 0;
constexpr uint32_t kStageOff = kQOff + kBM * kD * 2;
constexpr uint32_t kBarOff = kStageOff + kStages * kStageBytes;
constexpr uint32_t kNumBars = 18;  // 17 in use, rounded to keep the slot 16-byte aligned
constexpr uint32_t kSmemBytes = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kRescaleStep = 8.f;  // raise the running max only when it grows by > 2^8

// tensor-memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColPhi = 256;
constexpr uint32_t kColPlo = 320;
constexpr uint32_t kColO = 384;

struct TcParams {
    const int32_t* cu_q_lens;
    const int32_t* context_lens;
    const int32_t* block_tables;
    float* out;
    uint32_t* dev_status;
    int32_t Hq, Hkv, G, tq, P, num_pages, max_blocks, max_q_len, total_q;
    int32_t head_first;
    float scale_log2;
};

// Bounded wait that also gives up when another role has aborted.
__device__ inline bool wait_bar(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    return false;
}

__device__ inline void raise_abort(volatile uint32_t* abort_flag, uint32_t* dev_status) {
    *abort_flag = 1u;
    flag(dev_status, PA_DEV_TIMEOUT);
}

// hi/lo split of two probabilities into packed 16-bit pairs (low half = even key)
template <typename T> struct Pack;
template <> struct Pack<__nv_bfloat16> {
    __device__ static inline void split(float a, float b, uint32_t& hi, uint32_t& lo) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
};
template <> struct Pack<__half> {
    __device__ static inline void split(float a, float b, uint32_t& hi, uint32_t& lo) {
        const __half2 h = __floats2half2_rn(a, b);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const TcParams a) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const int g = blockIdx.x % a.Hkv, b = blockIdx.x / a.Hkv;
    const int tile = gridDim.y - 1 - blockIdx.y;  // heaviest row tiles first
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G, P = a.P;

    // ---- rows of this tile and their causal ends --------------------------------
    const int L = a.context_lens[b];
    const int row0 = a.cu_q_lens[b];
    const int Tq = a.cu_q_lens[b + 1] - row0;
    const bool bad = Tq < 0 || row0 < 0 || L < Tq || L > a.max_blocks * P || Tq > a.max_q_len;
    const int r_first = tile * a.tq;
    const int t_rows = max(0, min(Tq, a.max_q_len));
    const int n_rows =
        row0 < 0 ? 0 : max(0, min(min(a.tq, t_rows - r_first), a.total_q - (row0 + r_first)));
    if (bad && tile == 0 && tid == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
    if (n_rows <= 0) return;
    if (bad) {  // no key is read; the tile's rows are written as zeros
        for (int i = tid; i < n_rows * G * (kD / 4); i += kThreads) {
            const int r = i / (G * (kD / 4)), rest = i % (G * (kD / 4));
            const int h = rest / (kD / 4), c = rest % (kD / 4);
            float* o = a.out + (int64_t(row0 + r_first + r) * a.Hq + g * G + h) * kD;
            reinterpret_cast<float4*>(o)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    const int start = L - Tq;
    const int kend = start + r_first + n_rows;  // keys [0, kend) are visible to some row
    const int nt = (kend + kBN - 1) / kBN;
    const int npg = (kend + P - 1) / P;         // pages holding visible keys
    const int PT = kBN / P;                     // pages per key tile
    const int32_t* table = a.block_tables + int64_t(b) * a.max_blocks;

    // ---- shared memory ------------------------------------------------------------
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base + kQOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kBarOff);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* v_full = bars + 1 + kStages;
    uint64_t* kv_empty = bars + 1 + 2 * kStages;
    uint64_t* s_full = bars + 1 + 3 * kStages;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* o_done = p_full + 1;
    uint64_t* mma_done = o_done + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile uint32_t* abort_flag = tslot + 1;
    auto stage_k = [&](int st) { return base + kStageOff + st * kStageBytes; };
    auto stage_v = [&](int st) { return base + kStageOff + st * kStageBytes + kTileBytes; };

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        mbar_fence_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tslot;

    if (warp == 0) {
        // ================================ producer ================================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            // full box bytes count even where the box leaves the tensor (zero fill)
            mbar_arrive_expect_tx(q_full, 2u * 128u * uint32_t(G * a.tq));
            tma_load_3d(sQ, &tmQ, q_full, 0, g * G, row0 + r_first);
            tma_load_3d(sQ + kHalfBytes, &tmQ, q_full, 64, g * G, row0 + r_first);
            const int xc = a.head_first ? g : 0, yc = a.head_first ? 0 : g;
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int st = j % kStages;
                if (j >= kStages && !wait_bar(&kv_empty[st], ((j / kStages) - 1) & 1, abort_flag)) {
                    raise_abort(abort_flag, a.dev_status);
                    break;
                }
                int pg[8];
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const int idx = j * PT + p;
                    pg[p] = a.num_pages;  // beyond the tensor: the box reads as zeros
                    if (p < PT && idx < npg) {
                        const int e = table[idx];
                        if (e >= 0 && e < a.num_pages)
                            pg[p] = e;
                        else
                            flag(a.dev_status, PA_DEV_BAD_PAGE);
                    }
                }
                uint8_t* sK = stage_k(st);
                uint8_t* sV = stage_v(st);
                mbar_arrive_expect_tx(&k_full[st], kTileBytes);
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    if (p < PT)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            tma_load_4d(sK + hh * kHalfBytes + p * P * 128, &tmK, &k_full[st], 64 * hh, xc,
                                        yc, pg[p]);
                mbar_arrive_expect_tx(&v_full[st], kTileBytes);
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    if (p < PT)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            tma_load_4d(sV + hh * kHalfBytes + p * P * 128, &tmV, &v_full[st], 64 * hh, xc,
                                        yc, pg[p]);
                issued = j + 1;
            }
            // never leave the CTA with copies in flight
            for (int j = max(0, issued - kStages); j < issued; ++j) {
                const int st = j % kStages;
                mbar_wait(&k_full[st], (j / kStages) & 1, kWaitLimit);
                mbar_wait(&v_full[st], (j / kStages) & 1, kWaitLimit);
            }
            if (!mbar_wait(q_full, 0, kWaitLimit)) flag(a.dev_status, PA_DEV_TIMEOUT);
        }
    } else if (warp == 1) {
        // ================================== MMA ===================================
        if (lane == 0) {
            const uint32_t idQK = tc::idesc_f16(kBM, kBN, kBf16, false);
            const uint32_t idPV = tc::idesc_f16(kBM, kD, kBf16, true);
            const uint32_t q_addr = smem_u32(sQ);
            bool ok = wait_bar(q_full, 0, abort_flag);
            tc::fence_after_sync();
            auto pv = [&](int i) -> bool {
                const int st = i % kStages;
                if (!wait_bar(p_full, i & 1, abort_flag)) return false;
                if (!wait_bar(&v_full[st], (i / kStages) & 1, abort_flag)) return false;
                tc::fence_after_sync();
                const uint32_t v_addr = smem_u32(stage_v(st));
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks) {
                    // 16 keys: 8-row core groups 1024 B apart, dim halves 16 KB apart
                    const uint64_t bd = tc::smem_desc_sw128(v_addr + ks * 2048, kHalfBytes, 1024);
                    tc::mma_ts(tm + kColO, tm + kColPhi + ks * 8, bd, idPV, i > 0 || ks > 0);
                    tc::mma_ts(tm + kColO, tm + kColPlo + ks * 8, bd, idPV, true);
                }
                tc::commit(&kv_empty[st]);
                tc::commit(o_done);
                return true;
            };
            for (int j = 0; ok && j < nt; ++j) {
                const int st = j % kStages, sb = j & 1;
                ok = wait_bar(&k_full[st], (j / kStages) & 1, abort_flag);
                if (ok && j >= 2) ok = wait_bar(&s_free[sb], ((j - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc::fence_after_sync();
                const uint32_t k_addr = smem_u32(stage_k(st));
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                    tc::mma_ss(tm + kColS + sb * kBN, tc::smem_desc_sw128(q_addr + off, 16, 1024),
                               tc::smem_desc_sw128(k_addr + off, 16, 1024), idQK, ks > 0);
                }
                tc::commit(&s_full[sb]);
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok) ok = pv(nt - 1);
            if (!ok) raise_abort(abort_flag, a.dev_status);
            // every MMA issued so far has finished before tensor memory is freed
            tc::commit(mma_done);
            if (!mbar_wait(mma_done, 0, kWaitLimit)) flag(a.dev_status, PA_DEV_TIMEOUT);
        }
    } else {
        // ================================= softmax =================================
        const int quad = warp & 3;
        const int m = quad * 32 + lane;  // MMA row = tensor-memory lane
        const uint32_t lane_addr = uint32_t(quad * 32) << 16;
        const int t = m / G, h = m - (m / G) * G;
        const bool row_ok = t < a.tq && t < n_rows;
        const int lim = row_ok ? start + r_first + t + 1 : 0;  // keys [0, lim)
        const float sl2 = a.scale_log2;
        const int pshift = P == 16 ? 4 : 5;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        uint32_t s[4][32];
        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1, st = j % kStages, k0 = j * kBN;
            // pages of this tile outside the pool are skipped (flagged by the producer)
            bool pok = true;
            {
                const int idx = j * PT + lane;
                if (lane < PT && idx < npg) {
                    const int e = __ldg(table + idx);
                    pok = e >= 0 && e < a.num_pages;
                }
            }
            ok = __all_sync(0xffffffffu, wait_bar(&s_full[sb], (j >> 1) & 1, abort_flag));
            if (!ok) break;
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::ld_32x32b_x32(tm + lane_addr + kColS + sb * kBN + 32 * c, s[c]);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);
            const uint32_t pmask = __ballot_sync(0xffffffffu, pok);

            // scores in base-2 units, masked keys at -inf
            float mx = -INFINITY;
            if (k0 + kBN <= lim && pmask == 0xffffffffu) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float x = __uint_as_float(s[c][k]) * sl2;
                        s[c][k] = __float_as_uint(x);
                        mx = fmaxf(mx, x);
                    }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int key = k0 + 32 * c + k;
                        const bool vis = key < lim && ((pmask >> ((32 * c + k) >> pshift)) & 1u);
                        const float x = vis ? __uint_as_float(s[c][k]) * sl2 : -INFINITY;
                        s[c][k] = __float_as_uint(x);
                        mx = fmaxf(mx, x);
                    }
            }
            const bool need = mx > m_run + kRescaleStep;
            const float alpha = need ? ex2(m_run - mx) : 1.f;
            if (need) m_run = mx;
            l_run *= alpha;

            // O and the P buffer are free once PV_{j-1} has finished
            if (j > 0) {
                ok = __all_sync(0xffffffffu, wait_bar(o_done, (j - 1) & 1, abort_flag));
                if (!ok) break;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, need)) {
                    uint32_t o[32];
#pragma unroll 1
                    for (int c = 0; c < kD / 32; ++c) {
                        tc::ld_32x32b_x32(tm + lane_addr + kColO + 32 * c, o);
                        tc::wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tc::st_32x32b_x32(tm + lane_addr + kColO + 32 * c, o);
                    }
                }
            }

            // probabilities: p = 2^(x - m_run), split hi + lo, into tensor memory
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // keys 32c .. 32c+31 -> columns 16c .. 16c+15
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float p0 = ex2(__uint_as_float(s[c][2 * w]) - mu);
                    const float p1 = ex2(__uint_as_float(s[c][2 * w + 1]) - mu);
                    sum += p0 + p1;
                    Pack<T>::split(p0, p1, hi[w], lo[w]);
                }
                tc::st_32x32b_x16(tm + lane_addr + kColPhi + 16 * c, hi);
                tc::st_32x32b_x16(tm + lane_addr + kColPlo + 16 * c, lo);
            }
            l_run += sum;
            tc::wait_st();

            // slots past the context in its last page may hold anything (NaN):
            // zero those V rows so that 0 * V stays 0
            const int zlo = L - k0, zhi = min(kBN, npg * P - k0);
            if (zlo < zhi) {
                ok = __all_sync(0xffffffffu, wait_bar(&v_full[st], (j / kStages) & 1, abort_flag));
                if (!ok) break;
                uint8_t* sV = stage_v(st);
                for (int i = m; i < (zhi - zlo) * 16; i += kBM) {
                    const int row = zlo + (i >> 4), c = i & 15;
                    *reinterpret_cast<uint4*>(sV + (c >> 3) * kHalfBytes + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // ---- epilogue: O / l ------------------------------------------------------
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(o_done, (nt - 1) & 1, abort_flag));
        if (ok) {
            tc::fence_after_sync();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            float* orow = a.out + (int64_t(row0 + r_first + t) * a.Hq + g * G + h) * kD;
            uint32_t o[32];
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                tc::ld_32x32b_x32(tm + lane_addr + kColO + 32 * c, o);
                tc::wait_ld();
                if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(orow + 32 * c);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                             __uint_as_float(o[4 * k + 2]) * inv,
                                             __uint_as_float(o[4 * k + 3]) * inv);
                }
            }
        } else {
            raise_abort(abort_flag, a.dev_status);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
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

template <typename T>
cudaError_t launch_typed(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const TcParams& p,
                         int n_tiles, int B, cudaStream_t st) {
    auto kern = prefill_tc<T>;
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<dim3(p.Hkv * B, n_tiles), kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(pa_dtype dt, int D, int P, int G) {
    return dt != PA_F32 && D == kD && (P == 16 || P == 32) && G >= 1 && G <= kMaxGroup;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st) {
    if (!prefill_tc_supported(dt, D, P, a.group)) return cudaErrorInvalidValue;
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
    p.head_first = head_first;
    p.scale_log2 = a.scale_log2;
    const int n_tiles = (a.max_q_len + tq - 1) / tq;
    if (n_tiles > 65535 || int64_t(a.num_kv_heads) * a.num_seqs > 0x7fffffff) return cudaErrorInvalidValue;
    return dt == PA_BF16 ? launch_typed<__nv_bfloat16>(mq, mk, mv, p, n_tiles, a.num_seqs, st)
                         : launch_typed<__half>(mq, mk, mv, p, n_tiles, a.num_seqs, st);
}

}  // namespace pa
