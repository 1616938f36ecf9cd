// pa_prefill_f32.cu -- chunked causal prefill with fp32 Q/K/V on the CUDA
// cores, register-tiled.
//
// One CTA per (row tile, kv head, sequence).  A row tile is 64 distributions
// (row = token * G + head: 64/G consecutive chunk rows times the G q heads
// of one kv head), so every K/V row staged in shared memory serves all G
// heads and all of the tile's rows (minfer doc 71: the GQA-batched shape;
// crucible paged attention results: K/V shared across the q heads of one kv
// head and across query rows).  Keys come in blocks of 64, gathered page by
// page through the block table with 16-byte cp.async copies, one block in
// flight while the previous one is computed.
//
// Each of the 256 threads owns a 4 x 4 block of a key block's scores (4
// distributions, 4 keys 16 apart) and the same 4 distributions' rows of O
// (4 or 8 dims); probabilities pass to the P.V step through shared memory,
// transposed.  The softmax is online, in base 2 (q is pre-scaled by
// scale * log2 e), with the row max and the denominator reduced over the 16
// threads of a row group by shuffles in a fixed order.
// Row r of a chunk of T rows over a context of L keys sees keys 0..L-T+r
// (crucible README, "Prefill scheduling").
#include "pa_prefill_f32.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kM = 64;     // distributions per row tile
constexpr int kKB = 64;    // keys per block
constexpr int kThr = 256;  // 16 row groups x 16 threads

__device__ inline void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ inline void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ inline void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Sum / max over the 16 threads of a row group (lanes 0-15 or 16-31 of a
// warp), butterfly order: every thread of the group gets the same value.
__device__ inline float group_sum(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ inline float group_max(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int D> struct F32Tile {
    static constexpr int kLd = D + 4;           // padded row (floats)
    static constexpr int kQ = kM * kLd;         // Q tile (pre-scaled)
    static constexpr int kBlk = kKB * kLd;      // one K (or V) block
    static constexpr int kPld = kM + 4;         // row of P transposed: [key][distribution]
    static constexpr size_t kBytes =
        sizeof(float) * (size_t(kQ) + 4 * size_t(kBlk) + size_t(kKB) * kPld) + sizeof(int) * 2 * kKB;
};

template <int D, int P>
__global__ void __launch_bounds__(kThr, 1) prefill_f32(const AttnArgs a) {
    using S = F32Tile<D>;
    constexpr int kLd = S::kLd, kPld = S::kPld;
    constexpr int kDv = D / 64;                   // float4 columns of O a thread owns
    constexpr int kChunks = D / 4;                // 16-byte chunks of a K/V row
    constexpr int kCp = kKB * kChunks / kThr;     // K (and V) copies a thread issues per block
    extern __shared__ float4 smem4[];
    float* q_s = reinterpret_cast<float*>(smem4);
    float* kv_s = q_s + S::kQ;                    // [2 buffers][K, V][kKB][kLd]
    float* p_t = kv_s + 4 * S::kBlk;              // [kKB][kPld]
    int* ok_s = reinterpret_cast<int*>(p_t + kKB * kPld);  // [2 buffers][kKB]: key in a pool page

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    // grid (kv head x sequence, tile), tiles launched latest rows (most keys)
    // first across all (sequence, kv head) pairs, so a last partial wave
    // holds the lightest tiles
    const int g = int(blockIdx.x) % a.num_kv_heads, b = int(blockIdx.x) / a.num_kv_heads;
    const int tile = int(gridDim.y - 1 - blockIdx.y);
    const int G = a.group, Hq = a.num_q_heads;
    const int tq = kM / G;  // chunk rows of a tile

    pdl_launch_dependents();
    pdl_wait_primary();  // the previous kernel's writes are visible from here on

    // ---- rows of this tile and their causal ends ------------------------------
    const int L = PA_IN(b, a.num_seqs, a.dev_status) ? a.context_lens[b] : 0;
    const bool in = PA_IN(b + 1, a.num_seqs + 1, a.dev_status);
    const int row0 = in ? a.cu_q_lens[b] : 0;
    const int Tq = in ? a.cu_q_lens[b + 1] - row0 : 0;
    const bool bad = Tq < 0 || row0 < 0 || L < Tq || L > a.max_blocks_per_seq * P || Tq > a.max_q_len;
    if (bad && tile == 0 && tid == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
    const int r_first = tile * tq;
    const int t_rows = max(0, min(Tq, a.max_q_len));
    const int n_rows = row0 < 0 ? 0 : max(0, min(min(tq, t_rows - r_first), a.total_q - (row0 + r_first)));
    if (n_rows <= 0) return;  // the whole CTA, before any barrier
    const int start = L - Tq;
    const int kend = bad ? 0 : start + r_first + n_rows;  // keys [0, kend) are visible to some row
    const int nblk = (kend + kKB - 1) / kKB;              // bad: none, and the rows are written as zeros

    const float* kbase = static_cast<const float*>(a.k) + int64_t(g) * a.head_stride;
    const float* vbase = static_cast<const float*>(a.v) + int64_t(g) * a.head_stride;
    const int32_t* table = a.block_tables + int64_t(b) * a.max_blocks_per_seq;

    // Stage key block kb into buffer u: keys past kend, and keys of pages
    // outside the pool (flagged), become zero rows marked not ok.
    auto load_block = [&](int kb, int u) {
        float* ks = kv_s + 2 * u * S::kBlk;
        float* vs = ks + S::kBlk;
#pragma unroll
        for (int n = 0; n < kCp; ++n) {
            const int i = tid + n * kThr;
            const int j = i / kChunks, c = i % kChunks;
            const int key = kb * kKB + j;
            bool ok = false;
            int32_t pg = 0;
            if (key < kend && PA_IN(key / P, a.max_blocks_per_seq, a.dev_status)) {
                pg = table[key / P];
                ok = pg >= 0 && pg < a.num_pages;
                if (!ok && c == 0 && key % P == 0) flag(a.dev_status, PA_DEV_BAD_PAGE);
            }
            float* kd = ks + j * kLd + c * 4;
            float* vd = vs + j * kLd + c * 4;
            if (ok) {
                const int64_t off = int64_t(pg) * a.page_stride + int64_t(key % P) * a.token_stride + c * 4;
                cp16(kd, kbase + off);
                cp16(vd, vbase + off);
            } else {
                *reinterpret_cast<float4*>(kd) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(vd) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (c == 0) ok_s[u * kKB + j] = ok;
        }
        cp_commit();
    };
    if (nblk > 0) load_block(0, 0);  // in flight while q is staged

    // ---- Q tile, times scale * log2 e; distributions past the rows are zero ----
    for (int i = tid; i < kM * kChunks; i += kThr) {
        const int r = i / kChunks, c = i % kChunks;
        const int t = r / G, h = r - t * G;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < tq * G && t < n_rows) {
            const int64_t qi = (int64_t(row0 + r_first + t) * Hq + g * G + h) * D + c * 4;
            if (PA_IN(qi + 3, a.q_elems, a.dev_status)) {
                x = *reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + qi);
                x.x *= a.scale_log2;
                x.y *= a.scale_log2;
                x.z *= a.scale_log2;
                x.w *= a.scale_log2;
            }
        }
        *reinterpret_cast<float4*>(q_s + r * kLd + c * 4) = x;
    }

    // ---- this thread's four distributions --------------------------------------
    bool rok[4];  // the distribution is one of the tile's (row, head) pairs
    int endk[4];  // its last visible key (inclusive)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i, t = r / G;
        rok[i] = r < tq * G && t < n_rows;
        endk[i] = rok[i] && !bad ? start + r_first + t : -1;
    }
    float o[4][4 * kDv];
    float m_run[4], l_part[4];  // l_part: this thread's keys only, summed over the group at the end
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m_run[i] = -INFINITY;
        l_part[i] = 0.f;
#pragma unroll
        for (int e = 0; e < 4 * kDv; ++e) o[i][e] = 0.f;
    }

    for (int kb = 0; kb < nblk; ++kb) {
        const int u = kb & 1;
        if (kb + 1 < nblk) {
            load_block(kb + 1, u ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();  // block kb (and the q tile) in shared memory
        const float* ks = kv_s + 2 * u * S::kBlk;
        const float* vs = ks + S::kBlk;

        // ---- scores: s[i][k] = q(ty*4+i) . k(tx+16k) ---------------------------
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) s[i][k] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; d += 4) {
            float4 qv[4], kv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const float4*>(q_s + (ty * 4 + i) * kLd + d);
#pragma unroll
            for (int k = 0; k < 4; ++k) kv[k] = *reinterpret_cast<const float4*>(ks + (tx + 16 * k) * kLd + d);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    s[i][k] = fmaf(qv[i].x, kv[k].x, s[i][k]);
                    s[i][k] = fmaf(qv[i].y, kv[k].y, s[i][k]);
                    s[i][k] = fmaf(qv[i].z, kv[k].z, s[i][k]);
                    s[i][k] = fmaf(qv[i].w, kv[k].w, s[i][k]);
                }
        }

        // ---- mask, online softmax, P transposed into shared memory -------------
        bool kok[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) kok[k] = ok_s[u * kKB + tx + 16 * k] != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mb = -INFINITY;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int key = kb * kKB + tx + 16 * k;
                s[i][k] = (kok[k] && key <= endk[i]) ? s[i][k] : -INFINITY;
                mb = fmaxf(mb, s[i][k]);
            }
            const float m_new = fmaxf(m_run[i], group_max(mb));
            const float alpha = m_new == -INFINITY ? 1.f : ex2(m_run[i] - m_new);
            float ps = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[i][k] = m_new == -INFINITY ? 0.f : ex2(s[i][k] - m_new);
                ps += s[i][k];
            }
            l_part[i] = l_part[i] * alpha + ps;
            m_run[i] = m_new;
#pragma unroll
            for (int e = 0; e < 4 * kDv; ++e) o[i][e] *= alpha;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4*>(p_t + (tx + 16 * k) * kPld + ty * 4) =
                make_float4(s[0][k], s[1][k], s[2][k], s[3][k]);
        __syncthreads();  // P complete

        // ---- O += P V ---------------------------------------------------------
#pragma unroll 4
        for (int j = 0; j < kKB; ++j) {
            const float4 p = *reinterpret_cast<const float4*>(p_t + j * kPld + ty * 4);
#pragma unroll
            for (int v = 0; v < kDv; ++v) {
                const float4 w = *reinterpret_cast<const float4*>(vs + j * kLd + 64 * v + tx * 4);
                const float pr[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[i][4 * v + 0] = fmaf(pr[i], w.x, o[i][4 * v + 0]);
                    o[i][4 * v + 1] = fmaf(pr[i], w.y, o[i][4 * v + 1]);
                    o[i][4 * v + 2] = fmaf(pr[i], w.z, o[i][4 * v + 2]);
                    o[i][4 * v + 3] = fmaf(pr[i], w.w, o[i][4 * v + 3]);
                }
            }
        }
        __syncthreads();  // buffer u and P are rewritten by the next blocks
    }

    // ---- O / l: the denominator summed over the row group in a fixed order ------
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float l = group_sum(l_part[i]);
        if (!rok[i]) continue;  // an invalid length writes its rows as zeros (l = 0)
        const int r = ty * 4 + i, t = r / G, h = r - t * G;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t oi = (int64_t(row0 + r_first + t) * Hq + g * G + h) * D;
#pragma unroll
        for (int v = 0; v < kDv; ++v) {
            const int64_t at = oi + 64 * v + tx * 4;
            if (PA_IN(at + 3, a.out_elems, a.dev_status))
                *reinterpret_cast<float4*>(a.out + at) =
                    make_float4(o[i][4 * v] * inv, o[i][4 * v + 1] * inv, o[i][4 * v + 2] * inv, o[i][4 * v + 3] * inv);
        }
    }
}

template <int D, int P>
cudaError_t launch(const AttnArgs& a, cudaStream_t st) {
    auto k = prefill_f32<D, P>;
    const size_t sm = F32Tile<D>::kBytes;
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int tq = kM / a.group;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.num_kv_heads) * unsigned(a.num_seqs), unsigned((a.max_q_len + tq - 1) / tq));
    cfg.blockDim = dim3(kThr);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace

bool prefill_f32_supported(int D, int P, int G) {
    return (D == 64 || D == 128) && (P == 16 || P == 32) && G >= 1 && G <= kMaxGroup;
}

cudaError_t launch_prefill_f32(const AttnArgs& in, int D, int P, cudaStream_t st) {
    if (!prefill_f32_supported(D, P, in.group) || in.out == nullptr || in.cu_q_lens == nullptr)
        return cudaErrorInvalidValue;
    const int64_t tiles = (int64_t(in.max_q_len) + kM / in.group - 1) / (kM / in.group);
    if (int64_t(in.num_kv_heads) * in.num_seqs > 0x7fffffff || tiles > 65535) return cudaErrorInvalidValue;
    AttnArgs a = in;
    a.q_elems = a.out_elems = int64_t(a.total_q) * a.num_q_heads * D;
    if (D == 64) return P == 16 ? launch<64, 16>(a, st) : launch<64, 32>(a, st);
    return P == 16 ? launch<128, 16>(a, st) : launch<128, 32>(a, st);
}

}  // namespace pa
