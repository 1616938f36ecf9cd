// pa_tile_v0.cu -- first CUDA path: one CTA per (key split or row tile,
// kv head, sequence), all q heads of the kv head in the CTA so each K/V page
// row is read from HBM once per kv head (minfer doc 71: the GQA-batched
// shape; crucible results: one CTA shares K/V across the q heads of one kv
// head).  CUDA-core fp32 arithmetic, 16-byte page-row loads staged through
// registers one page ahead, online softmax per page (crucible results, the
// online-softmax experiment), base-2 exponentials.
//
// It serves four roles: the decode split partial (R = 1 row per sequence),
// the chunked-prefill kernel for the shapes the tensor-core and fp32
// prefill kernels do not take (R rows per tile, causal per row), the
// multi-row decode split partial (row tiles x key splits), and the fp32-KV
// decode path.  The split combine is at the end of this file.
#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kThreads = 128;

template <int D, int P, int R>
struct TileSmem {
    static constexpr int kDist = R * kMaxGroup;  // distributions (row, head)
    static constexpr int kGroups = kThreads / D; // threads sharing a dim
    static constexpr size_t bytes =
        sizeof(float) * (size_t(kDist) * D            // q (pre-scaled)
                         + size_t(P) * (D + 1)         // K page, padded rows
                         + size_t(P) * D               // V page
                         + size_t(kDist) * P           // scores / probabilities
                         + 3 * size_t(kDist));         // m, l, alpha
};

template <typename T, int D, int P, int R>
__global__ void __launch_bounds__(kThreads) attn_tile_v0(AttnArgs a) {
    using S = TileSmem<D, P, R>;
    constexpr int kVec = Elt<T>::kVec;
    constexpr int kChunks = D / kVec;  // 16-byte vectors per page row
    constexpr int kPerThread = S::kDist / S::kGroups;

    extern __shared__ float smem[];
    float* q_s = smem;
    float* k_s = q_s + S::kDist * D;
    float* v_s = k_s + P * (D + 1);
    float* p_s = v_s + P * D;
    float* m_s = p_s + S::kDist * P;
    float* l_s = m_s + S::kDist;
    float* al_s = l_s + S::kDist;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.z, g = blockIdx.y;
    const int G = a.group, Hq = a.num_q_heads;
    const bool fixed_rows = a.cu_q_lens == nullptr && a.rows_per_seq > 1;  // multi-row decode
    const bool decode = a.cu_q_lens == nullptr && !fixed_rows;
    // Split partials: x indexes the key split (one row), or row tile x split
    // for several rows per sequence; a direct pass has one split.
    const int Sn = a.out == nullptr ? a.num_splits : 1;
    const int split = decode ? blockIdx.x : blockIdx.x % Sn;
    const int tile = decode ? 0 : blockIdx.x / Sn;

    pdl_launch_dependents();
    pdl_wait_primary();  // the previous kernel's writes are visible from here on

    // ---- rows of this tile and their causal ends --------------------------
    int L = PA_IN(b, a.num_seqs, a.dev_status) ? a.context_lens[b] : 0;
    int row0, Tq;  // first packed row, rows of this sequence
    if (decode) {
        row0 = b;
        Tq = 1;
    } else if (fixed_rows) {
        row0 = b * a.rows_per_seq;
        Tq = a.rows_per_seq;
    } else {
        const bool in = PA_IN(b + 1, a.num_seqs + 1, a.dev_status);
        row0 = in ? a.cu_q_lens[b] : 0;
        Tq = in ? a.cu_q_lens[b + 1] - row0 : 0;
    }
    const bool bad = (Tq < 0) || (row0 < 0) || (L < Tq) || (L > a.max_blocks_per_seq * P) ||
                     (!decode && Tq > a.max_q_len);
    if (bad) {
        if (tid == 0 && blockIdx.x == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
        L = 0;  // no key is read; the tile's rows are written as zeros
    }
    const int start = L - Tq;
    const int r_first = tile * R;
    // rows of this tile that exist: below T (and the host bound), inside q/out
    int n_rows = 1;
    if (!decode) {
        const int t_rows = max(0, min(Tq, a.max_q_len));
        n_rows = row0 < 0 ? 0 : max(0, min(min(R, t_rows - r_first), a.total_q - (row0 + r_first)));
    }
    const int nd = R * G;

    // key range [t0, t1): up to the tile's last causal end, cut to the split
    int t0 = 0, t1 = decode ? L : ((n_rows > 0 && !bad) ? start + r_first + n_rows : 0);
    if (a.out == nullptr) {
        t0 = split * a.split_tokens;  // a whole number of pages
        t1 = min(t1, t0 + a.split_tokens);
    }

    const T* kbase = static_cast<const T*>(a.k) + int64_t(g) * a.head_stride;
    const T* vbase = static_cast<const T*>(a.v) + int64_t(g) * a.head_stride;
    const int32_t* table = a.block_tables + int64_t(b) * a.max_blocks_per_seq;

    // Page rows of kv head g travel through registers: every 16-byte load of
    // a page is issued before the first one is used, and the next page's
    // loads are in flight while this page is computed.
    constexpr int kLd = (P * kChunks + kThreads - 1) / kThreads;  // loads per thread, K and V each
    uint4 kr[kLd], vr[kLd];
    auto valid = [&](int32_t pg) { return pg >= 0 && pg < a.num_pages; };  // uniform across the CTA
    auto fetch = [&](int32_t pg, int ps) {
        const int n = min(P, t1 - ps);
#pragma unroll
        for (int u = 0; u < kLd; ++u) {
            const int i = tid + u * kThreads;
            if (i < n * kChunks) {
                const int j = i / kChunks, c = i % kChunks;
                const int64_t off = int64_t(pg) * a.page_stride + int64_t(j) * a.token_stride + c * kVec;
                kr[u] = *reinterpret_cast<const uint4*>(kbase + off);
                vr[u] = *reinterpret_cast<const uint4*>(vbase + off);
            }
        }
    };
    // The first table entry does not wait for the length: its index is known.
    const int32_t first = t0 / P < a.max_blocks_per_seq && PA_IN(t0 / P, a.max_blocks_per_seq, a.dev_status)
                              ? table[t0 / P]
                              : -1;
    int32_t next = t0 < t1 ? first : -1;
    if (t0 < t1 && valid(next)) fetch(next, t0);  // in flight while q is staged

    // ---- stage q (times scale*log2e) and reset the running state ----------
    for (int i = tid; i < nd * D; i += kThreads) {
        const int dist = i / D, d = i % D, r = dist / G, h = dist % G;
        float x = 0.f;
        if (r < n_rows) {
            const int64_t qi = (int64_t(row0 + r_first + r) * Hq + g * G + h) * D + d;
            if (PA_IN(qi, a.q_elems, a.dev_status)) x = Elt<T>::f(static_cast<const T*>(a.q)[qi]) * a.scale_log2;
        }
        q_s[dist * D + d] = x;
    }
    for (int i = tid; i < nd; i += kThreads) {
        m_s[i] = -INFINITY;
        l_s[i] = 0.f;
    }
    float acc[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) acc[k] = 0.f;
    const int my_d = tid % D, my_grp = tid / D;
    __syncthreads();

    for (int ps = t0; ps < t1; ps += P) {
        const int n = min(P, t1 - ps);
        const int32_t page = next;
        if (valid(page)) {  // -- registers -> shared (fp32)
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int i = tid + u * kThreads;
                if (i < n * kChunks) {
                    const int j = i / kChunks, c = i % kChunks;
                    float f[kVec];
                    vec_to_f32<T>(kr[u], f);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) k_s[j * (D + 1) + c * kVec + e] = f[e];
                    vec_to_f32<T>(vr[u], f);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) v_s[j * D + c * kVec + e] = f[e];
                }
            }
        }
        next = ps + P < t1 && PA_IN((ps + P) / P, a.max_blocks_per_seq, a.dev_status) ? table[(ps + P) / P] : -1;
        if (!valid(page)) {
            if (tid == 0) flag(a.dev_status, PA_DEV_BAD_PAGE);
            if (ps + P < t1 && valid(next)) fetch(next, ps + P);
            continue;
        }
        __syncthreads();
        if (ps + P < t1 && valid(next)) fetch(next, ps + P);
        // -- scores (base-2 units), masked per row's causal end
        for (int i = tid; i < nd * P; i += kThreads) {
            const int dist = i / P, j = i % P, r = dist / G;
            const int key = ps + j;
            const int end = start + r_first + r;  // inclusive
            float s = -INFINITY;
            if (j < n && r < n_rows && key <= end) {
                float dot = 0.f;
                const float* qd = q_s + dist * D;
                const float* kd = k_s + j * (D + 1);
#pragma unroll 8
                for (int d = 0; d < D; ++d) dot = fmaf(qd[d], kd[d], dot);
                s = dot;
            }
            p_s[dist * P + j] = s;
        }
        __syncthreads();
        // -- online softmax update, one warp per distribution
        for (int dist = warp; dist < nd; dist += kThreads / 32) {
            const float x = lane < P ? p_s[dist * P + lane] : -INFINITY;
            const float m_old = m_s[dist];
            const float m_new = fmaxf(m_old, warp_max(x));
            float p = 0.f, alpha = 1.f;
            if (m_new != -INFINITY) {
                p = ex2(x - m_new);
                alpha = ex2(m_old - m_new);
            }
            const float sum = warp_sum(p);
            if (lane < P) p_s[dist * P + lane] = p;
            if (lane == 0) {
                l_s[dist] = l_s[dist] * alpha + sum;
                m_s[dist] = m_new;
                al_s[dist] = alpha;
            }
        }
        __syncthreads();
        // -- rescale and accumulate P.V
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int dist = my_grp + k * S::kGroups;
            if (dist < nd) {
                float x = acc[k] * al_s[dist];
                const float* pr = p_s + dist * P;
                for (int j = 0; j < n; ++j) x = fmaf(pr[j], v_s[j * D + my_d], x);
                acc[k] = x;
            }
        }
        __syncthreads();
    }

    // ---- outputs -------------------------------------------------------------
    if (a.out == nullptr) {  // split partial of each (row, q head): (m, l) and the unscaled sum
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int dist = my_grp + k * S::kGroups;
            if (dist < nd) {
                const int r = dist / G, h = dist % G;
                if (r < n_rows) {
                    const int64_t idx = (int64_t(row0 + r_first + r) * Hq + g * G + h) * Sn + split;
                    if (!PA_IN(idx, a.partial_items, a.dev_status)) continue;
                    if (m_s[dist] != -INFINITY) a.partial_acc[idx * D + my_d] = acc[k];
                    if (my_d == 0) {
                        a.partial_ml[idx * 2] = m_s[dist];
                        a.partial_ml[idx * 2 + 1] = l_s[dist];
                    }
                }
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int dist = my_grp + k * S::kGroups;
            if (dist < nd) {
                const int r = dist / G, h = dist % G;
                if (r < n_rows) {
                    const float l = l_s[dist];
                    const int64_t oi = (int64_t(row0 + r_first + r) * Hq + g * G + h) * D + my_d;
                    if (PA_IN(oi, a.out_elems, a.dev_status)) a.out[oi] = l > 0.f ? acc[k] / l : 0.f;
                }
            }
        }
    }
}

// Combine: one CTA per (q head, sequence), one thread per output dim.  The
// partials are [B][Hq][S][...]; sequence b merges its first S_b splits, S_b =
// splits_per_seq[b] clamped to [0, S] (all S when splits_per_seq is NULL).
__global__ void combine_v0(const float* __restrict__ ml, const float* __restrict__ acc,
                           float* __restrict__ out, int Hq, int S, int D,
                           const int32_t* __restrict__ splits_per_seq) {
    // Batches of 32 splits: lane j holds split x0 + j's (m, l), every thread
    // loads its dim of all 32 accumulators at once; batches are merged by
    // rescaling in ascending split order (fixed shuffle trees, no atomics).
    constexpr int kB = 32;
    pdl_launch_dependents();
    pdl_wait_primary();  // the partials are complete from here on
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x, lane = d & 31;
    const int64_t base = (int64_t(b) * Hq + h) * S;
    const int Sb = splits_per_seq ? min(max(splits_per_seq[b], 0), S) : S;  // splits of this sequence
    float M = -INFINITY, num = 0.f, den = 0.f;
    for (int x0 = 0; x0 < Sb; x0 += kB) {
        const int cnt = min(kB, Sb - x0);
        float mj = -INFINITY, lj = 0.f;
        if (lane < cnt) {
            const float2 v = *reinterpret_cast<const float2*>(ml + (base + x0 + lane) * 2);
            mj = v.x;
            lj = v.y;
        }
        float av[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) av[j] = j < cnt ? acc[(base + x0 + j) * D + d] : 0.f;
        const float Mn = fmaxf(M, warp_max(mj));
        if (Mn == -INFINITY) continue;  // no key so far
        const float sc = ex2(M - Mn);   // M = -inf -> 0
        const float w = mj == -INFINITY ? 0.f : ex2(mj - Mn);
        den = den * sc + warp_sum(w * lj);
        num *= sc;
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
            num = wj != 0.f ? fmaf(wj, av[j], num) : num;  // an empty split's acc is never written
        }
        M = Mn;
    }
    out[(int64_t(b) * Hq + h) * D + d] = den > 0.f ? num / den : 0.f;
}

template <typename T, int D, int P, int R>
cudaError_t launch_one(const AttnArgs& a, dim3 grid, cudaStream_t st) {
    auto k = attn_tile_v0<T, D, P, R>;
    const size_t sm = TileSmem<D, P, R>::bytes;
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // Programmatic dependent launch: the CTAs may start while the previous
    // kernel finishes; the kernel waits for it before reading global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <typename T, int R>
cudaError_t dispatch_dp(const AttnArgs& a, int D, int P, dim3 grid, cudaStream_t st) {
    if (D == 64 && P == 16) return launch_one<T, 64, 16, R>(a, grid, st);
    if (D == 64 && P == 32) return launch_one<T, 64, 32, R>(a, grid, st);
    if (D == 128 && P == 16) return launch_one<T, 128, 16, R>(a, grid, st);
    if (D == 128 && P == 32) return launch_one<T, 128, 32, R>(a, grid, st);
    return cudaErrorInvalidValue;
}

template <int R>
cudaError_t dispatch_t(const AttnArgs& a, pa_dtype dt, int D, int P, dim3 grid, cudaStream_t st) {
    switch (dt) {
    case PA_F32: return dispatch_dp<float, R>(a, D, P, grid, st);
    case PA_F16: return dispatch_dp<__half, R>(a, D, P, grid, st);
    case PA_BF16: return dispatch_dp<__nv_bfloat16, R>(a, D, P, grid, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

namespace {
// The buffers' extents (total_q rows of Hq x D; split partials per row and
// q head), for the checked build's range checks.
AttnArgs with_extents(const AttnArgs& in, int D) {
    AttnArgs a = in;
    a.q_elems = a.out_elems = int64_t(a.total_q) * a.num_q_heads * D;
    a.partial_items = int64_t(a.total_q) * a.num_q_heads * (a.num_splits > 0 ? a.num_splits : 1);
    return a;
}
}  // namespace

cudaError_t launch_decode_v0(const AttnArgs& in, pa_dtype dt, int D, int P, cudaStream_t st) {
    const AttnArgs a = with_extents(in, D);
    dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
    return dispatch_t<1>(a, dt, D, P, grid, st);
}

cudaError_t launch_prefill_v0(const AttnArgs& in, pa_dtype dt, int D, int P, cudaStream_t st) {
    const AttnArgs a = with_extents(in, D);
    constexpr int R = 4;
    const int splits = a.out == nullptr ? a.num_splits : 1;  // split partials: multi-row decode only
    if (splits < 1 || (splits > 1 && a.cu_q_lens != nullptr)) return cudaErrorInvalidValue;
    dim3 grid((a.max_q_len + R - 1) / R * splits, a.num_kv_heads, a.num_seqs);
    return dispatch_t<R>(a, dt, D, P, grid, st);
}

cudaError_t launch_combine_v0(const float* ml, const float* acc, float* out, int B, int Hq,
                              int S, int D, cudaStream_t st, const int32_t* splits_per_seq) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hq, B);
    cfg.blockDim = dim3(D);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_v0, ml, acc, out, Hq, S, D, splits_per_seq);
}

namespace {
// One CTA per sequence: the Hkv rows of its new token go to row L - 1 of
// page block_tables[b][(L - 1) / P]; E is an unsigned type of the element size.
template <typename E>
__global__ void append_kv(const E* __restrict__ k_new, const E* __restrict__ v_new, E* k, E* v,
                          const int32_t* __restrict__ bt, const int32_t* __restrict__ cl, int Hkv, int D, int P,
                          int num_pages, int max_blocks, int64_t ps, int64_t ts, int64_t hs) {
    const int b = blockIdx.x;
    const int L = cl[b];
    if (L < 1 || L > max_blocks * P) return;  // the attention flags it
    const int pg = bt[(int64_t)b * max_blocks + (L - 1) / P];
    if (pg < 0 || pg >= num_pages) return;
    const int64_t row = (int64_t)pg * ps + (int64_t)((L - 1) % P) * ts;
    for (int i = threadIdx.x; i < Hkv * D; i += blockDim.x) {
        const int g = i / D, d = i - g * D;
        k[row + g * hs + d] = k_new[((int64_t)b * Hkv + g) * D + d];
        v[row + g * hs + d] = v_new[((int64_t)b * Hkv + g) * D + d];
    }
}
}  // namespace

cudaError_t launch_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens, int B, int Hkv,
                             int D, int P, int elt_bytes, int num_pages, int max_blocks, int64_t page_stride,
                             int64_t token_stride, int64_t head_stride, cudaStream_t st) {
    const int threads = Hkv * D < 1024 ? Hkv * D : 1024;
    if (elt_bytes == 4)
        append_kv<uint32_t><<<B, threads, 0, st>>>(
            static_cast<const uint32_t*>(k_new), static_cast<const uint32_t*>(v_new), static_cast<uint32_t*>(k_cache),
            static_cast<uint32_t*>(v_cache), block_tables, context_lens, Hkv, D, P, num_pages, max_blocks,
            page_stride, token_stride, head_stride);
    else
        append_kv<uint16_t><<<B, threads, 0, st>>>(
            static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), static_cast<uint16_t*>(k_cache),
            static_cast<uint16_t*>(v_cache), block_tables, context_lens, Hkv, D, P, num_pages, max_blocks,
            page_stride, token_stride, head_stride);
    return cudaGetLastError();
}

}  // namespace pa
