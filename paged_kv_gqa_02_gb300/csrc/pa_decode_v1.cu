// pa_decode_v1.cu -- decode attention for 16-bit K/V on sm_103a.
//
// Work partition (split-KV, crucible README "Split-position attention";
// minfer doc 71: all q heads of a kv head share each K/V tile).  The work of
// a call is the ordered list of (sequence, kv head) units, unit (b, g) made of
// the pages of sequence b read for kv head g.  In a cost space where each
// unit occupies unit_cost + pages positions (unit_cost stands for the fixed
// work of a unit piece: its query rows and its result), the grid's
// n = min(CTAs x 8 warps, T / kMinPartCost) parts take equal contiguous shares
// [v*T/n, (v+1)*T/n).  Every warp therefore moves about the same
// number of bytes whatever the mix of context lengths, and the grid does not
// depend on device data.  A warp finishes a unit that lies inside its share;
// the pieces of the other units go to the workspace and a combine kernel,
// launched with programmatic dependent launch, merges them in ascending part
// order (split-KV combine, crucible README "Split-position attention":
// rescale by exp(m_i - m_max), then merge).
//
// Each warp reads the block table of its share ahead (32 pages at a time,
// one lane per page) and issues its own TMA copies of each page's K and V
// tiles (one kv head, all page_size slots, 128B-swizzled) into its own ring
// of half-stages guarded by mbarriers, refilling a slot as soon as it has
// used it; no warp waits for another.  Each warp streams its pages: S = Q K^T with
// mma.sync m16n8k16 (the group's q heads padded to 16 rows), an online softmax
// in base 2 (crucible results, the online-softmax experiment), and O += P V
// with m16n8k16 whose A operand is built from the S accumulator in registers.
// The probabilities are split into a 16-bit high part and a 16-bit remainder
// stacked along k (the V fragment is passed twice), keeping 16 (bf16) or 22
// (f16) bits of them: one 16-bit rounding alone moves small outputs by more
// than 1% of their size.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kCW = 8;                        // warps per CTA, each a partition part
constexpr int kThreadsV1 = kCW * 32;
constexpr uint32_t kWaitLimit = 1u << 22;     // polls before a wait gives up
constexpr int kMaxTiles = 64;                 // page tiles (half-stages) per CTA, at most
constexpr int kMaxRing = 16;                  // page tiles in one warp's ring, at most
constexpr int kSmemLimit = 232448;            // 227 KiB opt-in per CTA
constexpr int kUnitCost = 2;                  // partition weight of a unit piece, in pages
constexpr int kMinPartCost = 4;               // smallest share worth a warp, in cost units

struct V1Params {
    const void* q;  // [B*Hq][D]
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* out;
    float* ws_ml;   // [slot][G][2]
    float* ws_acc;  // [slot][G][D]
    uint32_t* dev_status;
    int32_t B, Hq, Hkv, G, num_pages, max_blocks, max_len;
    float scale_log2;
    int32_t n_parts, ntiles, head_first, unit_cost;
};

// A warp's position in its share of the cost space.
struct Walk {
    long long start, s, e;  // cost position of the unit's first slot; share [s, e)
    int b, g, pb, pf, pe;   // unit, its pages, the pages [pf, pe) of it in the share
    int done;
};

__host__ __device__ inline size_t v1_fixed_bytes() {
    return size_t(kMaxTiles) * 4      // page id of each tile
           + size_t(kMaxTiles) * 8;   // a full barrier per tile
}

__device__ inline int pages_of_len(int L, int P, int max_len) {
    return (L >= 1 && L <= max_len) ? (L + P - 1) / P : 0;
}

__device__ inline int seq_pages(const int32_t* cl, int b, int P, int max_len) {
    return pages_of_len(__ldg(cl + b), P, max_len);
}

__device__ inline long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ inline long long warp_incl_scan_ll(long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Total cost T of the call (all units with pages).  Whole warp.
__device__ inline long long total_cost(const V1Params& a, int P) {
    long long tot = 0;
    for (int b = threadIdx.x & 31; b < a.B; b += 32) {
        const int pb = seq_pages(a.context_lens, b, P, a.max_len);
        if (pb > 0) tot += (long long)a.Hkv * (pb + a.unit_cost);
    }
    return warp_sum_ll(tot);
}

// The walk of share [s, e): its first unit piece.  Whole warp.
__device__ inline Walk walk_start(const V1Params& a, int P, long long s, long long e) {
    const int lane = threadIdx.x & 31, W = a.unit_cost;
    Walk w{0, s, e, 0, 0, 0, 0, 0, 1};
    if (e <= s) return w;
    long long basep = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const int pb = b < a.B ? seq_pages(a.context_lens, b, P, a.max_len) : 0;
        const long long c = pb > 0 ? (long long)a.Hkv * (pb + W) : 0;
        const long long incl = warp_incl_scan_ll(c, lane);
        const long long total = __shfl_sync(0xffffffffu, incl, 31);
        if (s < basep + total) {
            const unsigned m = __ballot_sync(0xffffffffu, basep + incl > s);
            const int j = __ffs(m) - 1;
            const long long seq0 = basep + __shfl_sync(0xffffffffu, incl - c, j);
            w.pb = __shfl_sync(0xffffffffu, pb, j);
            w.b = b0 + j;
            w.g = int((s - seq0) / (w.pb + W));
            w.start = seq0 + (long long)w.g * (w.pb + W);
            const long long pf = s - w.start - W > 0 ? s - w.start - W : 0;
            const long long room = e - w.start - W;
            const long long pe = room < w.pb ? room : w.pb;
            w.pf = int(pf);
            w.pe = int(pe);
            w.done = pe <= pf;
            return w;
        }
        basep += total;
    }
    return w;
}

// Moves to the next unit with pages; done once its pages start at or after e.
__device__ inline void walk_next_unit(Walk& w, const V1Params& a, int P) {
    w.start += w.pb + a.unit_cost;
    if (++w.g == a.Hkv) {
        w.g = 0;
        int pb = 0;
        do {
            ++w.b;
        } while (w.b < a.B && (pb = seq_pages(a.context_lens, w.b, P, a.max_len)) == 0);
        if (w.b >= a.B) {
            w.done = 1;
            return;
        }
        w.pb = pb;
    }
    w.pf = 0;
    const long long room = w.e - w.start - a.unit_cost;
    w.pe = int(room < w.pb ? room : w.pb);
    if (w.pe <= 0) w.done = 1;
}

// Advances the walk by j pages; `i` is the current page within the unit.
__device__ inline void walk_advance(Walk& w, int& i, int j, const V1Params& a, int P) {
    while (!w.done && j > 0) {
        const int rem = w.pe - i;
        if (j < rem) {
            i += j;
            j = 0;
        } else {
            j -= rem;
            walk_next_unit(w, a, P);
            i = w.pf;
        }
    }
}

// Splits two probabilities into 16-bit high parts and 16-bit remainders,
// packed as the pairs an MMA A-fragment register holds.
template <typename T>
__device__ inline void split_hi_lo(float x, float y, uint32_t& hi, uint32_t& lo) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        const float2 f = __bfloat1622float2(h);
        const __nv_bfloat162 r = __floats2bfloat162_rn(x - f.x, y - f.y);
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&r);
    } else {
        const __half2 h = __floats2half2_rn(x, y);
        const float2 f = __half22float2(h);
        const __half2 r = __floats2half2_rn(x - f.x, y - f.y);
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&r);
    }
}

// Part v of the partition runs on CTA v % n_ctas, warp v / n_ctas, so that
// when fewer parts than warps are in use every SM still gets a share.  The
// number of parts in use is a function of the inputs alone.
__device__ inline long long parts_in_use(long long T, const V1Params& a) {
    const long long want = (T + kMinPartCost - 1) / kMinPartCost;
    return want < 1 ? 1 : (want < a.n_parts ? want : a.n_parts);
}

// The load side of a warp: lane l holds page base + l of the warp's share
// (its kv head, page id and whether it exists).
struct LoadWindow {
    Walk w;     // walk state at page `base` of the share
    int i;      // page within the unit at `base`
    int base;   // share page index of lane 0
    int live, g, page;
};

__device__ inline void window_fill(LoadWindow& lw, const V1Params& a, int P) {
    Walk x = lw.w;
    int i = lw.i;
    walk_advance(x, i, threadIdx.x & 31, a, P);
    lw.live = x.done ? 0 : 1;
    lw.g = x.g;
    lw.page = lw.live ? __ldg(a.block_tables + (long long)x.b * a.max_blocks + i) : -1;
}

// At most 224 registers a thread: 256 x 224 leaves room on the SM for one
// combine CTA, which then starts (and locates its items) while this grid runs.
template <typename T, int D, int P, int NT>
__global__ void __maxnreg__(224)
    decode_v1(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const V1Params a) {
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kHalves = D / 64;     // 128-byte swizzle spans per row
    constexpr int kTile = P * D * 2;    // one K (or V) page tile: a half-stage
    constexpr int kMt = P / 16;         // 16-key row blocks of a page
    constexpr int kKs = D / 16;         // k-steps of K Q^T; 16-dim row blocks of O^T

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_launch_dependents();

    // ---- this warp's share of the cost space ------------------------------------
    const long long cost = total_cost(a, P);
    const long long n_used = parts_in_use(cost, a);
    const long long part = (long long)warp * gridDim.x + blockIdx.x;
    if (part >= n_used) return;
    // The CTA's pool of page tiles is divided among its active warps
    // (warps 0 .. active-1), so a CTA with few parts keeps more pages in
    // flight per part.
    const int active = int((n_used - blockIdx.x + gridDim.x - 1) / gridDim.x);
    const int NH = min(a.ntiles / active, kMaxRing);
    uint8_t* my_tiles = base + size_t(warp) * NH * kTile;  // [NH][kTile]
    int* my_page = reinterpret_cast<int*>(base + size_t(a.ntiles) * kTile) + warp * NH;
    uint64_t* my_full =
        reinterpret_cast<uint64_t*>(reinterpret_cast<int*>(base + size_t(a.ntiles) * kTile) + kMaxTiles) +
        warp * NH;
    if (lane == 0) {
        for (int s = 0; s < NH; ++s) mbar_init(&my_full[s], 1);
        mbar_fence_init();
        if (warp == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
    }
    __syncwarp();
    Walk wk = walk_start(a, P, part * cost / n_used, (part + 1) * cost / n_used);
    if (wk.done) return;

    // ---- load side: issue half-stage x (page x/2 of the share; K, then V)
    LoadWindow lw{wk, wk.pf, 0, 0, 0, -1};
    window_fill(lw, a, P);
    bool timed_out = false;
    auto issue = [&](int hx) {
        const int j = hx >> 1;
        while (j >= lw.base + 32) {  // next 32 pages of the share
            walk_advance(lw.w, lw.i, 32, a, P);
            lw.base += 32;
            window_fill(lw, a, P);
        }
        const int src = j - lw.base;
        const int live = __shfl_sync(0xffffffffu, lw.live, src);
        const int g = __shfl_sync(0xffffffffu, lw.g, src);
        const int pg = __shfl_sync(0xffffffffu, lw.page, src);
        if (!live) return;
        if (lane == 0) {
            const int slot = hx % NH;
            const bool ok = pg >= 0 && pg < a.num_pages;
            if (!ok && (hx & 1) == 0) flag(a.dev_status, PA_DEV_BAD_PAGE);
            my_page[slot] = ok ? pg : -1;
            mbar_arrive_expect_tx(&my_full[slot], ok ? kTile : 0);
            if (ok) {
                uint8_t* dst = my_tiles + size_t(slot) * kTile;
                const int xc = a.head_first ? g : 0, yc = a.head_first ? 0 : g;
#pragma unroll
                for (int hh = 0; hh < kHalves; ++hh)
                    tma_load_4d(dst + hh * P * 128, (hx & 1) ? &tmV : &tmK, &my_full[slot], 64 * hh, xc, yc,
                                pg);
            }
        }
        __syncwarp();
    };
    for (int hx = 0; hx < NH; ++hx) issue(hx);  // fill the ring

    // ---- compute side: S^T = K Q^T and O^T += V^T P^T ---------------------------
    // Keys (for S^T) and head dims (for O^T) are the MMA rows; the group's q
    // heads are its 8-wide columns (NT column tiles), so a group of G <= 8
    // heads wastes at most half of each MMA.
    const int g4 = lane >> 2, t4 = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: the matrix and row this lane addresses
    const int G = a.G;
    // Byte offset of (row, 16-byte chunk) in a page tile: two 64-dim halves of
    // P rows of 128 bytes, chunks XOR-swizzled by row (128-byte swizzle).
    auto swz = [](int row, int chunk) -> uint32_t {
        return uint32_t((chunk >> 3) * (P * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
    };
    uint32_t offK[kKs], offV[kKs];
#pragma unroll
    for (int j = 0; j < kKs; ++j) {
        offK[j] = swz((lm & 1) * 8 + lr, 2 * j + (lm >> 1));  // A = K rows (keys) x dims 16j..
        offV[j] = swz((lm >> 1) * 8 + lr, 2 * j + (lm & 1));  // A = V^T rows (dims 16j..) x keys
    }
    uint32_t qb[NT][kKs][2], qn[NT][kKs][2];
    float o[kKs][NT][4];
    float sc[kMt][NT][4];
    // B fragments of Q^T for unit (b, g): column n = q head nt*8 + g4 (0 past G)
    auto load_q = [&](uint32_t (&dst)[NT][kKs][2], int b, int g) {
        const T* qbase = static_cast<const T*>(a.q) + ((long long)b * a.Hq + g * G) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + g4;
            const uint32_t* row = reinterpret_cast<const uint32_t*>(qbase + (h < G ? h : 0) * D);
#pragma unroll
            for (int ks = 0; ks < kKs; ++ks) {
                dst[nt][ks][0] = h < G ? __ldg(row + 8 * ks + t4) : 0u;
                dst[nt][ks][1] = h < G ? __ldg(row + 8 * ks + 4 + t4) : 0u;
            }
        }
    };
    load_q(qn, wk.b, wk.g);
    int x = 0;  // half-stage number

    while (!wk.done) {
        const int L = __ldg(a.context_lens + wk.b);
        const bool whole = (wk.pf == 0) && (wk.pe == wk.pb);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ks = 0; ks < kKs; ++ks) {
                qb[nt][ks][0] = qn[nt][ks][0];
                qb[nt][ks][1] = qn[nt][ks][1];
            }
        Walk nx = wk;  // the next piece, whose query rows load now
        walk_next_unit(nx, a, P);
        if (!nx.done) load_q(qn, nx.b, nx.g);

        // running max and (lane-partial) denominator of heads nt*8 + 2*t4 + j
        float mrun[NT][2], lrun[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mrun[nt][0] = mrun[nt][1] = -INFINITY;
            lrun[nt][0] = lrun[nt][1] = 0.f;
        }
#pragma unroll
        for (int dt = 0; dt < kKs; ++dt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) o[dt][nt][0] = o[dt][nt][1] = o[dt][nt][2] = o[dt][nt][3] = 0.f;

        for (int i = wk.pf; i < wk.pe; ++i) {
            const int ntok = min(P, L - i * P);
            // ---- K tile: S^T = K Q^T, masked, online softmax
            bool ok = !timed_out;
            if (ok && !mbar_wait(&my_full[x % NH], (x / NH) & 1, kWaitLimit)) {
                timed_out = true;
                ok = false;
                if (lane == 0) flag(a.dev_status, PA_DEV_TIMEOUT);
            }
            const bool valid = ok && my_page[x % NH] >= 0;
            if (valid) {
                const uint32_t kb = smem_u32(my_tiles + size_t(x % NH) * kTile);
#pragma unroll
                for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) sc[mt][nt][0] = sc[mt][nt][1] = sc[mt][nt][2] = sc[mt][nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kKs; ++ks) {
#pragma unroll
                    for (int mt = 0; mt < kMt; ++mt) {
                        uint32_t ka[4];
                        ldsm_x4(kb + mt * 2048 + offK[ks], ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) mma_16816<kBf>(sc[mt][nt], ka, qb[nt][ks][0], qb[nt][ks][1]);
                    }
                }
            }
            __syncwarp();
            if (!timed_out) issue(x + NH);  // the K slot is free again
            ++x;
            uint32_t ph[kMt][NT][2], pl[kMt][NT][2];  // P^T as B fragments: high parts, remainders
            if (valid) {
                float mx[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
                for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = 16 * mt + g4 + ((e & 2) ? 8 : 0);
                            const float v = tok < ntok ? sc[mt][nt][e] * a.scale_log2 : -INFINITY;
                            sc[mt][nt][e] = v;
                            mx[nt][e & 1] = fmaxf(mx[nt][e & 1], v);
                        }
                bool same = true;
                float al[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float v = mx[nt][j];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        const float mn = fmaxf(mrun[nt][j], v);
                        al[nt][j] = ex2(mrun[nt][j] - mn);  // m = -inf -> 0
                        same = same && al[nt][j] == 1.f;
                        mrun[nt][j] = mn;
                        lrun[nt][j] *= al[nt][j];
                    }
#pragma unroll
                for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            sc[mt][nt][e] = ex2(sc[mt][nt][e] - mrun[nt][e & 1]);
                            lrun[nt][e & 1] += sc[mt][nt][e];
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            uint32_t hi, lo;
                            split_hi_lo<T>(sc[mt][nt][2 * j], sc[mt][nt][2 * j + 1], hi, lo);
                            ph[mt][nt][j] = movm_trans(hi);
                            pl[mt][nt][j] = movm_trans(lo);
                        }
                    }
                if (!__all_sync(0xffffffffu, same)) {
#pragma unroll
                    for (int dt = 0; dt < kKs; ++dt)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            o[dt][nt][0] *= al[nt][0];
                            o[dt][nt][1] *= al[nt][1];
                            o[dt][nt][2] *= al[nt][0];
                            o[dt][nt][3] *= al[nt][1];
                        }
                }
            }
            // ---- V tile: O^T += V^T P^T
            ok = !timed_out;
            if (ok && !mbar_wait(&my_full[x % NH], (x / NH) & 1, kWaitLimit)) {
                timed_out = true;
                ok = false;
                if (lane == 0) flag(a.dev_status, PA_DEV_TIMEOUT);
            }
            if (valid && ok) {
                uint8_t* vt = my_tiles + size_t(x % NH) * kTile;
                if (ntok < P) {  // rows past the context hold arbitrary bits: zero them
                    for (int y = lane; y < (P - ntok) * kHalves * 8; y += 32) {
                        const int rowi = ntok + y / (kHalves * 8);
                        const int rem = y % (kHalves * 8);
                        *reinterpret_cast<uint4*>(vt + (rem >> 3) * (P * 128) + rowi * 128 + (rem & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const uint32_t vb = smem_u32(vt);
#pragma unroll
                for (int kk = 0; kk < kMt; ++kk)
#pragma unroll
                    for (int dt = 0; dt < kKs; ++dt) {
                        uint32_t va[4];
                        ldsm_x4_t(vb + kk * 2048 + offV[dt], va[0], va[1], va[2], va[3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_16816<kBf>(o[dt][nt], va, ph[kk][nt][0], ph[kk][nt][1]);
                            mma_16816<kBf>(o[dt][nt], va, pl[kk][nt][0], pl[kk][nt][1]);
                        }
                    }
            }
            __syncwarp();
            if (!timed_out) issue(x + NH);  // the V slot is free again
            ++x;
        }

        // ---- the piece's result: final output, or a partial for the combine.
        // Lane (g4, t4) holds dims 16*dt + g4 (+8) of heads nt*8 + 2*t4 + j.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = lrun[nt][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                lrun[nt][j] = v;
            }
        if (whole) {
            float* ob = a.out + ((long long)wk.b * a.Hq + wk.g * G) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int h = nt * 8 + 2 * t4 + j;
                    if (h < G) {
                        const float inv = lrun[nt][j] > 0.f ? 1.f / lrun[nt][j] : 0.f;
#pragma unroll
                        for (int dt = 0; dt < kKs; ++dt) {
                            ob[h * D + 16 * dt + g4] = o[dt][nt][j] * inv;
                            ob[h * D + 16 * dt + g4 + 8] = o[dt][nt][2 + j] * inv;
                        }
                    }
                }
        } else {
            const long long slot = part + (long long)wk.b * a.Hkv + wk.g;
            float* accp = a.ws_acc + slot * G * D;
            float* ml = a.ws_ml + slot * G * 2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int h = nt * 8 + 2 * t4 + j;
                    if (h < G) {
#pragma unroll
                        for (int dt = 0; dt < kKs; ++dt) {
                            accp[h * D + 16 * dt + g4] = o[dt][nt][j];
                            accp[h * D + 16 * dt + g4 + 8] = o[dt][nt][2 + j];
                        }
                        if (g4 == 0) *reinterpret_cast<float2*>(ml + h * 2) = make_float2(mrun[nt][j], lrun[nt][j]);
                    }
                }
        }
        wk = nx;
    }
    // A wait that gave up may leave copies in flight: wait (bounded) for them.
    if (timed_out && lane == 0)
        for (int s = 0; s < NH; ++s) mbar_wait(&my_full[s], ((x + s) / NH) & 1, 1024);
}

// Merges the pieces of units that span several parts: one CTA per (sequence,
// q head), one thread per output dim.  The CTA locates its pieces from the
// lengths alone (a lane-parallel prefix over the sequences) before it waits
// for the partial kernel through programmatic dependent launch; after the
// wait, the (m, l) pairs of up to 32 pieces (one per lane) and their
// accumulators (one per thread and piece) are loaded together, so a merge
// costs about one L2 round trip.  Maxima and denominators are reduced by
// fixed shuffle trees and the accumulators are summed in ascending part
// order, so the result does not depend on timing.  At most 64 registers a
// thread (1024/D CTAs an SM), so the CTAs that start while the partial kernel
// runs fit beside its 256 x 224-register CTA.
template <int D>
__global__ void __launch_bounds__(D, 1024 / D) combine_v1(const V1Params a, int P) {
    constexpr int kBatch = 32;  // pieces loaded together
    const int lane = threadIdx.x & 31, d = threadIdx.x;
    const int item = blockIdx.x;  // b * Hq + h
    const int b = item / a.Hq, h = item % a.Hq, g = h / a.G, r = h % a.G;
    const int unit = b * a.Hkv + g;
    const int W = a.unit_cost;
    long long T = 0, pre = 0;
    for (int x = lane; x < a.B; x += 32) {
        const int pg = seq_pages(a.context_lens, x, P, a.max_len);
        const long long c = pg > 0 ? (long long)a.Hkv * (pg + W) : 0;
        T += c;
        if (x < b) pre += c;
    }
    T = warp_sum_ll(T);
    pre = warp_sum_ll(pre);
    const int pb = seq_pages(a.context_lens, b, P, a.max_len);
    const long long n = parts_in_use(T > 0 ? T : 1, a);
    long long c0 = 0;
    int np = 0;
    if (pb > 0) {  // the unit's pages sit at cost positions [p0, p0 + pb)
        const long long p0 = pre + (long long)g * (pb + W) + W;
        c0 = ((p0 + 1) * n - 1) / T;  // part v owns [v*T/n, (v+1)*T/n)
        const long long c1 = ((p0 + pb) * n - 1) / T;
        np = c1 > c0 ? int(c1 - c0 + 1) : 0;  // 0: finished inside one part
    }
    pdl_wait_primary();  // the partial kernel's pieces are complete from here on
    float* o = a.out + (long long)item * D + d;
    if (pb == 0) {
        *o = 0.f;
        if (h == 0 && d == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
        return;
    }
    if (np == 0) return;
    // Parts between c0 and c1 whose share is empty (possible when T < n) wrote
    // nothing: their weight is 0 and their rows are never used.
    float M = -INFINITY, den = 0.f, num = 0.f;
    for (int x0 = 0; x0 < np; x0 += kBatch) {
        const int cnt = min(kBatch, np - x0);
        float mj = -INFINITY, lj = 0.f;
        if (lane < cnt) {
            const long long cc = c0 + x0 + lane;
            if (cc * T / n != (cc + 1) * T / n) {
                const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + ((cc + unit) * a.G + r) * 2);
                mj = ml.x;
                lj = ml.y;
            }
        }
        const float* accp = a.ws_acc + ((c0 + x0 + unit) * a.G + r) * D + d;
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) v[j] = j < cnt ? accp[(long long)j * a.G * D] : 0.f;
        const float Mn = fmaxf(M, warp_max(mj));
        if (Mn == -INFINITY) continue;  // no key so far
        const float sc = ex2(M - Mn);   // M = -inf -> 0
        const float wj = mj == -INFINITY ? 0.f : ex2(mj - Mn);
        den = den * sc + warp_sum(wj * lj);
        num *= sc;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const float w = __shfl_sync(0xffffffffu, wj, j);
            num = w != 0.f ? fmaf(w, v[j], num) : num;
        }
        M = Mn;
    }
    *o = den > 0.f ? num / den : 0.f;
}

// ---- host side -------------------------------------------------------------------

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

// Page tiles per CTA: as many K/V page tiles as shared memory holds once a
// combine CTA (static shared memory and the per-CTA reservation) has room.
int tile_count(int D, int P) {
    const size_t tile = size_t(P) * D * 2;
    const size_t room = size_t(kSmemLimit) - 1024 - v1_fixed_bytes() - 2048;
    const int n = int(room / tile);
    return n > kMaxTiles ? kMaxTiles : n;
}

size_t smem_bytes(int D, int P, int ntiles) {
    return 1024 + size_t(ntiles) * P * D * 2 + v1_fixed_bytes();
}

template <typename T, int D, int P, int NT>
cudaError_t launch_partial(const CUtensorMap& k, const CUtensorMap& v, const V1Params& a, int n_ctas,
                           cudaStream_t st) {
    auto kern = decode_v1<T, D, P, NT>;
    static bool configured = false;  // benign race: every caller sets the same value
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<n_ctas, kThreadsV1, smem_bytes(D, P, a.ntiles), st>>>(k, v, a);
    return cudaGetLastError();
}

template <typename T, int D, int P>
cudaError_t launch_typed(const CUtensorMap& k, const CUtensorMap& v, const V1Params& a, int n_ctas,
                         int phases, cudaStream_t st) {
    if (phases & 1) {
        // one 8-wide column tile of q heads when the group fits, else two
        cudaError_t e = a.G <= 8 ? launch_partial<T, D, P, 1>(k, v, a, n_ctas, st)
                                 : launch_partial<T, D, P, 2>(k, v, a, n_ctas, st);
        if (e != cudaSuccess) return e;
    }
    if (!(phases & 2)) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.B) * unsigned(a.Hq));
    cfg.blockDim = dim3(D);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_v1<D>, a, P);
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: (m, l) pairs, then accumulators, one slot per (part, unit) piece.
struct WsLayout {
    size_t ml, acc, total;
};
WsLayout ws_layout(int B, int Hq, int Hkv, int D, int n_ctas) {
    const size_t slots = size_t(n_ctas) * kCW + size_t(B) * Hkv;
    const size_t G = size_t(Hq / Hkv);
    WsLayout w;
    w.ml = 0;
    w.acc = w.ml + round256(slots * G * 2 * sizeof(float));
    w.total = w.acc + slots * G * D * sizeof(float);
    return w;
}

}  // namespace

size_t decode_v1_workspace_bytes(int B, int Hq, int Hkv, int D, int n_ctas) {
    return ws_layout(B, Hq, Hkv, D, n_ctas).total;
}

cudaError_t launch_decode_v1(const DecodeV1Call& call, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int D = call.D, P = call.P;
    const CUtensorMapDataType dt =
        call.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // The pool as a 4-d tensor (head_dim, kv head, slot, page), the two middle
    // dimensions in stride order; the box is one page of one kv head, 64 dims
    // (128 bytes, the swizzle span) at a time.
    const int head_first = call.head_stride <= call.token_stride;
    CUtensorMap mk, mv;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    dims[0] = D;
    dims[3] = cuuint64_t(call.num_pages);
    strides[2] = cuuint64_t(call.page_stride) * 2;
    if (head_first) {
        dims[1] = call.Hkv;
        dims[2] = P;
        strides[0] = cuuint64_t(call.head_stride) * 2;
        strides[1] = cuuint64_t(call.token_stride) * 2;
        box[0] = 64; box[1] = 1; box[2] = P; box[3] = 1;
    } else {
        dims[1] = P;
        dims[2] = call.Hkv;
        strides[0] = cuuint64_t(call.token_stride) * 2;
        strides[1] = cuuint64_t(call.head_stride) * 2;
        box[0] = 64; box[1] = P; box[2] = 1; box[3] = 1;
    }
    if (enc(&mk, dt, 4, const_cast<void*>(call.k), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (enc(&mv, dt, 4, const_cast<void*>(call.v), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    V1Params a;
    a.q = call.q;
    a.block_tables = call.block_tables;
    a.context_lens = call.context_lens;
    a.out = call.out;
    const int G = call.Hq / call.Hkv;
    const WsLayout wl = ws_layout(call.B, call.Hq, call.Hkv, D, call.n_ctas);
    char* ws = static_cast<char*>(call.workspace);
    a.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    a.ws_acc = reinterpret_cast<float*>(ws + wl.acc);
    a.dev_status = call.dev_status;
    a.B = call.B;
    a.Hq = call.Hq;
    a.Hkv = call.Hkv;
    a.G = G;
    a.num_pages = call.num_pages;
    a.max_blocks = call.max_blocks;
    a.max_len = call.max_blocks * P;
    a.scale_log2 = call.scale_log2;
    a.n_parts = call.n_ctas * kCW;
    a.ntiles = tile_count(D, P);
    a.head_first = head_first;
    a.unit_cost = kUnitCost;
    if (a.ntiles < 2 * kCW) return cudaErrorInvalidValue;
    const bool bf = call.dtype == PA_BF16;
#define PA_V1_CASE(DD, PP)                                                                        \
    if (D == DD && P == PP)                                                                       \
        return bf ? launch_typed<__nv_bfloat16, DD, PP>(mk, mv, a, call.n_ctas, call.phases, st) \
                  : launch_typed<__half, DD, PP>(mk, mv, a, call.n_ctas, call.phases, st);
    PA_V1_CASE(128, 32)
    PA_V1_CASE(128, 16)
    PA_V1_CASE(64, 32)
    PA_V1_CASE(64, 16)
#undef PA_V1_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pa
