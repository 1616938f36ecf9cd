// pa_decode_v1.cu -- decode attention for 16-bit K/V on sm_103a.
//
// Work partition (split-KV, crucible README "Split-position attention";
// minfer doc 71: all q heads of a kv head share each K/V tile).  The work of
// a call is the ordered list of (sequence, kv head) units, unit (b, g) made of
// the pages of sequence b read for kv head g (with several query rows, one
// unit per row block of a kv head).  In a cost space where each
// unit occupies unit_cost + pages positions (unit_cost stands for the fixed
// work of a unit piece: its query row and its result), the n CTAs in use
// (all of the persistent grid unless the call is tiny) take equal contiguous
// shares [c*T/n, (c+1)*T/n), and the 8 warps of a CTA split its share the
// same way (fewer warps in small calls without the in-CTA merge).  Every
// working warp therefore moves about the same number of bytes
// whatever the mix of context lengths, and the grid does not depend on
// device data.  A warp finishes a unit that lies inside its part.  When the
// group's q heads fit one 8-wide MMA column tile, the warps of a CTA then
// merge the pieces they share in shared memory, so a unit leaves at most one
// piece per CTA; otherwise each warp writes its pieces.  A combine kernel,
// launched with programmatic dependent launch, merges the pieces of units
// that span several parts in ascending part order (split-KV combine, crucible
// README "Split-position attention": rescale by exp(m_i - m_max), then merge).
//
// Each warp reads the block table of its part ahead (32 pages at a time,
// one lane per page) and issues its own TMA copies of each page's K and V
// tiles (one kv head, all page_size slots, 128B-swizzled) into its own ring
// of half-stages guarded by mbarriers, refilling a slot as soon as it has
// used it; no warp waits for another.  Each warp streams its pages: S^T = K Q^T
// with mma.sync m16n8k16 (keys as the MMA rows, the group's q heads as its
// 8-wide columns), an online softmax in base 2 (crucible results, the
// online-softmax experiment), and O^T += V^T P^T with P^T moved into the B
// operand layout by movmatrix.  The probabilities are split into a 16-bit
// high part and a 16-bit remainder, both multiplied by V, keeping 16 (bf16)
// or 22 (f16) bits of them: one 16-bit rounding alone moves small outputs by
// more than 1% of their size.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kCW = 8;                        // warps per CTA, each a partition part
constexpr int kThreadsV1 = kCW * 32;
constexpr uint64_t kWaitNs = 2000000000ull;   // a wait gives up after 2 s of the global timer
constexpr int kMaxTiles = 64;                 // page tiles (half-stages) per CTA, at most
constexpr int kMaxRing = 16;                  // page tiles in one warp's ring, at most
constexpr int kSmemLimit = 232448;            // 227 KiB opt-in per CTA
constexpr int kUnitCost = 2;                  // partition weight of a unit piece, in pages
constexpr int kMinCtaCost = 3;                // smallest share worth a CTA, in cost units
constexpr int kCtaMergeMaxShare = 16;         // CTA merge only while CTA shares average at most this
// Single launch: a unit split over CTAs c0 .. c1 counts its pieces on counter
// c0 (each CTA boundary is crossed by at most one unit), so the counters take
// a fixed block at the start of the workspace whatever the call's sizes.
constexpr int kMaxCounters = int(PA_DECODE_COUNTER_BYTES / sizeof(unsigned));
constexpr int kDeadPage = -2;  // static plan: a page past the sequence's length (skipped, not an error)

struct V1Params {
    const void* q;  // [B*Hq][D]
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* out;
    float* ws_ml;   // [slot][G][2]
    float* ws_acc;  // [slot][G][D]
    unsigned* ws_cnt;  // [kMaxCounters] arrival counters, zero between calls
    long long ws_slots;               // pieces the workspace holds
    long long q_rows, out_rows;       // [B][T][Hq] rows of D in q and out (this launch's T)
    uint32_t* dev_status;
    int32_t B, Hq, Hkv, G, num_pages, max_blocks, max_len;
    int32_t window;     // > 0: a row sees only its last `window` keys
    // > 0 (small calls): the partition counts every sequence at this many
    // pages, so it follows from host parameters alone and a warp loads its
    // lengths and table entries in one round trip; pages past a sequence's
    // length are skipped (their ring slots are armed with no bytes)
    int32_t static_pages;
    int32_t debug_timeout;  // 1: each warp's first wait (on a barrier no copy targets) gives up at once
    int32_t T, t0, Gq;  // query rows per sequence, first row of this launch, q heads per kv head
    // Row blocks: the launch's Tl rows come in NB blocks of rb rows (the last
    // may be shorter), each block its own unit.  Unit (b, u), u < Hv = Hkv * NB,
    // reads kv head u / NB for rows t0 + (u % NB) * rb ...; its column c
    // (c < G = rb * Gq) is row t0 + (u % NB) * rb + c / Gq, q head
    // (u / NB) * Gq + c % Gq.
    int32_t Tl, rb, NB, Hv;
    float scale_log2;
    int32_t n_ctas, ntiles, unit_cost;
    int32_t cta_pieces;  // 1: the group fits one MMA column tile, so small calls merge per CTA
    // 1: single launch (asked for by the caller).  Every call merges its
    // warps' pieces per CTA, and the last CTA to leave a piece of a unit
    // merges that unit's CTA pieces, so no combine kernel runs (one column
    // tile, head_dim <= 128 only)
    int32_t finish;
    // KV append (nullptr: none): the new token of sequence b, kv head g is
    // row L_b - 1 of the cache; it is written there and used in place of the
    // row the page copy brought in
    const void* k_new;  // [B][Hkv][D]
    const void* v_new;
    void* k_cache;
    void* v_cache;
    int64_t page_stride, token_stride, head_stride;  // elements
};

// Append: puts the new token's row (kv head g of sequence b) into row `row`
// of a staged page tile (swizzled like the TMA copy) and into the cache.
// Lanes 0 .. D/8 - 1 move one 16-byte chunk each.
template <int D, int P>
__device__ inline void append_row(uint8_t* tile, const void* src_all, void* cache, const V1Params& a, int b,
                                  int g, int pg, int row) {
    const int lane = threadIdx.x & 31;
    if (lane < D / 8 && PA_IN((long long)b * a.Hkv + g, (long long)a.B * a.Hkv, a.dev_status)) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src_all) +
                                                             ((long long)b * a.Hkv + g) * D) +
                              lane);
        const int c8 = lane & 7;
        *reinterpret_cast<uint4*>(tile + (lane >> 3) * (P * 128) + row * 128 + ((c8 ^ (row & 7)) << 4)) = v;
        uint16_t* dst = static_cast<uint16_t*>(cache) + (long long)pg * a.page_stride +
                        (long long)row * a.token_stride + (long long)g * a.head_stride;
        reinterpret_cast<uint4*>(dst)[lane] = v;
    }
    fence_proxy_async_smem();  // the tile is a TMA destination again later
    __syncwarp();
}

__device__ inline int pages_of_len(int L, int P, int max_len, int T) {
    return (L >= T && L >= 1 && L <= max_len) ? (L + P - 1) / P : 0;
}

// First page holding a key that a row of this launch sees (sliding window;
// the launch's first row has the lowest window).
__device__ inline int first_page(const V1Params& a, int L, int P) {
    if (a.window <= 0) return 0;
    const int lo = L - a.T + a.t0 - a.window + 1;
    return lo > 0 ? lo / P : 0;
}

// Pages of sequence b in the work partition: its own (seq_pages) or, with
// a static plan, the same count for every sequence.
__device__ inline int part_pages(const V1Params& a, int b, int P);

// Kv head, first row and columns of unit u (a row block of a kv head).
__device__ inline int unit_head(const V1Params& a, int u) { return a.NB == 1 ? u : u / a.NB; }
__device__ inline int unit_row0(const V1Params& a, int u) { return a.NB == 1 ? a.t0 : a.t0 + (u % a.NB) * a.rb; }
__device__ inline int unit_cols(const V1Params& a, int u) {
    return a.NB == 1 ? a.G : min(a.rb, a.Tl - (u % a.NB) * a.rb) * a.Gq;
}

// Pages of sequence b that the unit reads (0: invalid length, fewer keys
// than query rows): from first_page to the page of key L - 1.
__device__ inline int seq_pages(const V1Params& a, int b, int P) {
    const int L = PA_IN(b, a.B, a.dev_status) ? __ldg(a.context_lens + b) : 0;
    const int n = pages_of_len(L, P, a.max_len, a.T);
    return n > 0 ? n - first_page(a, L, P) : 0;
}

__device__ inline int part_pages(const V1Params& a, int b, int P) {
    return a.static_pages > 0 ? a.static_pages : seq_pages(a, b, P);
}

// Offset (elements) of column c of unit (b, u) in q and out: [B][T][Hq][D].
template <int D>
__device__ inline long long row_off(const V1Params& a, int b, int u, int c) {
    const int tl = c / a.Gq;
    return (((long long)b * a.T + unit_row0(a, u) + tl) * a.Hq + (long long)unit_head(a, u) * a.Gq +
            (c - tl * a.Gq)) * D;
}

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
        const int pb = part_pages(a, b, P);
        if (pb > 0) tot += (long long)a.Hv * (pb + a.unit_cost);
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
        const int pb = b < a.B ? part_pages(a, b, P) : 0;
        const long long c = pb > 0 ? (long long)a.Hv * (pb + W) : 0;
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
    if (++w.g == a.Hv) {
        w.g = 0;
        int pb = 0;
        do {
            ++w.b;
        } while (w.b < a.B && (pb = part_pages(a, w.b, P)) == 0);
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

// CTAs that take a share: all of them unless the call is so small that a
// share would fall below kMinCtaCost.  A function of the inputs and the grid
// alone.  CTA c owns [c*T/n, (c+1)*T/n) of the cost space; its warp w owns
// the matching eighth, part c*8 + w of the n*8 warp parts (or, with wpc
// working warps a CTA, the matching wpc-th, part c*wpc + w).
__device__ inline long long ctas_in_use(long long T, long long grid) {
    const long long want = (T + kMinCtaCost - 1) / kMinCtaCost;
    return want < 1 ? 1 : (want < grid ? want : grid);
}

// Warps of each CTA that take a part when warps leave their own pieces: all
// eight unless the cost space is shorter than that, then about one per cost
// position (rounded up, so at most n_cta - 1 parts are empty), which spares
// the combine the mostly empty pieces of eight parts a CTA.  A function of
// the inputs and the grid alone.
__device__ inline int warps_in_use(long long T, long long n_cta) {
    const long long w = (T + n_cta - 1) / n_cta;
    return int(w < 1 ? 1 : (w > kCW ? kCW : w));
}

// Single launch: merges the np CTA pieces of unit u (slots c0 + u ..
// c0 + np - 1 + u, written by other CTAs of this grid) into the final rows,
// rescaling each by 2^(m_i - M) and summing in ascending CTA order.  Every
// thread of the CTA takes (head, 4 dims) items; the pieces are read through
// L2 (ld.global.cg) in batches whose loads are all in flight together.
template <int D>
__device__ __noinline__ void finish_unit(const V1Params& a, int u, int c0, int np) {
    constexpr int kB = 16;  // pieces loaded together
    const int G = a.G, ub = u / a.Hv, ug = u % a.Hv, Gu = unit_cols(a, ug);
    for (int idx = threadIdx.x; idx < G * D / 4; idx += kThreadsV1) {
        const int h = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
        float M = -INFINITY, den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < np; j0 += kB) {
            float2 ml[kB];
            float4 v[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                if (j0 + j < np && PA_IN((long long)c0 + j0 + j + u, a.ws_slots, a.dev_status)) {
                    const long long slot = (long long)c0 + j0 + j + u;
                    ml[j] = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + (slot * G + h) * 2));
                    v[j] = __ldcg(reinterpret_cast<const float4*>(a.ws_acc + (slot * G + h) * D + d4));
                } else {
                    ml[j] = make_float2(-INFINITY, 0.f);
                    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float Mn = M;
#pragma unroll
            for (int j = 0; j < kB; ++j) Mn = fmaxf(Mn, ml[j].x);
            if (Mn == -INFINITY) continue;  // no key so far
            const float sc = ex2(M - Mn);   // M = -inf -> 0
            den *= sc;
            num.x *= sc;
            num.y *= sc;
            num.z *= sc;
            num.w *= sc;
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                if (ml[j].x == -INFINITY) continue;  // an empty piece: weight 0
                const float w = ex2(ml[j].x - Mn);
                den = fmaf(w, ml[j].y, den);
                num.x = fmaf(w, v[j].x, num.x);
                num.y = fmaf(w, v[j].y, num.y);
                num.z = fmaf(w, v[j].z, num.z);
                num.w = fmaf(w, v[j].w, num.w);
            }
            M = Mn;
        }
        if (h < Gu && PA_IN(row_off<D>(a, ub, ug, h) / D, a.out_rows, a.dev_status)) {
            const float inv = den > 0.f ? 1.f / den : 0.f;
            *reinterpret_cast<float4*>(a.out + row_off<D>(a, ub, ug, h) + d4) =
                make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
        }
    }
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
    if (a.static_pages > 0) {
        // Static plan: the length and the table entry load together (entries
        // up to max_blocks lie in the caller's table row; one past the
        // sequence's pages is never used, and its page never read).
        const bool in = lw.live && PA_IN(i, a.max_blocks, a.dev_status);
        const int e = in ? __ldg(a.block_tables + (long long)x.b * a.max_blocks + i) : -1;
        const int L = lw.live ? __ldg(a.context_lens + x.b) : 0;
        const int n = pages_of_len(L, P, a.max_len, a.T);
        if (lw.live && n == 0 && i == 0 && x.g == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
        lw.page = !in ? -1 : (i < n ? e : kDeadPage);
        return;
    }
    const int fpg = lw.live ? first_page(a, __ldg(a.context_lens + x.b), P) : 0;
    lw.page = lw.live && PA_IN(fpg + i, a.max_blocks, a.dev_status)
                  ? __ldg(a.block_tables + (long long)x.b * a.max_blocks + fpg + i)
                  : -1;
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
    // One column tile: warps of a CTA merge their pieces in shared memory.
    // Two: each warp's non-whole pieces go to the workspace.
    constexpr bool kCtaMerge = NT == 1 && D <= 128;  // D 256: per-warp pieces (registers)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up that touches no global memory: it may overlap the kernel
    // before this one (programmatic dependent launch) ----------------------------
    int* tile_page = reinterpret_cast<int*>(base + size_t(a.ntiles) * kTile);  // [kMaxTiles]
    uint64_t* tile_full = reinterpret_cast<uint64_t*>(tile_page + kMaxTiles);  // [kMaxTiles]
    __shared__ int s_unit[kCW][2];  // CTA merge: unit of each warp's pieces (-1: none)
    __shared__ int s_inside[kCW][2];
    __shared__ long long s_p0[kCW][2];  // CTA merge: cost position of the unit's first page
    __shared__ int s_pb[kCW][2];        // and its page count
    __shared__ int4 s_run[2 * kCW];     // CTA merge: (unit, entry mask, inside, first entry) of each run
    __shared__ float s_w[kCtaMerge ? 8 : 1][2 * kCW];  // CTA merge: weight of each entry, per head
    __shared__ float s_md[kCtaMerge ? 8 : 1][2];       // CTA merge: max and denominator, per head
    __shared__ __align__(8) uint64_t s_never;  // a barrier no copy or thread ever arrives on (debug_timeout)
    __shared__ int2 s_fin[2 * kCW];     // single launch: (unit, first CTA) of each run this CTA completes
    __shared__ int s_fnp[2 * kCW];      // and its CTA pieces
    if (threadIdx.x < 2 * kCW) s_fin[threadIdx.x] = make_int2(-1, 0);
    if (lane == 0) {
        if constexpr (kCtaMerge) {  // eight rings, each warp initialises its own
            const int nh = min(a.ntiles / kCW, kMaxRing);
            for (int s = 0; s < nh; ++s) mbar_init(&tile_full[warp * nh + s], 1);
        } else {  // rings are cut once the call's size is known: every tile's barrier
            for (int s = warp; s < a.ntiles; s += kCW) mbar_init(&tile_full[s], 1);
        }
        if (warp == 0) mbar_init(&s_never, 1);
        mbar_fence_init();
        if (warp == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        s_unit[warp][0] = s_unit[warp][1] = -1;
    }
    __syncwarp();
    pdl_wait_primary();  // the previous kernel's writes are visible from here on
    // Only now may the combine kernel start: it reads the lengths before its
    // own wait, and they are complete once the kernel before this one is.
    pdl_launch_dependents();

    // ---- this CTA's share of the cost space, and this warp's part of it ---------
    const long long cost = total_cost(a, P);
    const long long n_cta = ctas_in_use(cost, gridDim.x);
    if (blockIdx.x >= n_cta) return;  // the whole CTA, before any CTA barrier
    const long long cta_s = (long long)blockIdx.x * cost / n_cta, cta_e = (blockIdx.x + 1) * cost / n_cta;
    // Small calls (short shares, few pages a warp) merge the warps' pieces in
    // the CTA, so the combine sees one piece per CTA; larger ones leave each
    // warp's pieces to the combine.  Uniform over the grid.
    const bool cta_merge = kCtaMerge && (a.finish || cost <= (long long)kCtaMergeMaxShare * n_cta);
    // Warps that take a part: with the CTA merge compiled in, a call past it
    // has shares above 16 and all eight do.
    const int wpc = kCtaMerge ? kCW : warps_in_use(cost, n_cta);
    const long long n = n_cta * wpc;
    const long long part = (long long)blockIdx.x * wpc + warp;
    const int NH = min(a.ntiles / wpc, kMaxRing);  // ring depth of a working warp
    const int ring = warp < wpc ? warp : 0;        // idle warps touch no ring
    uint8_t* my_tiles = base + size_t(ring) * NH * kTile;  // [NH][kTile]
    int* my_page = tile_page + ring * NH;
    uint64_t* my_full = tile_full + ring * NH;
    if constexpr (!kCtaMerge) __syncthreads();  // every tile barrier is initialised
    Walk wk = warp < wpc ? walk_start(a, P, part * cost / n, (part + 1) * cost / n)
                         : Walk{0, 0, 0, 0, 0, 0, 0, 0, 1};

    // ---- load side: issue half-stage x (page x/2 of the share; K, then V)
    // K/V are read once per call: evict-first keeps the kernel's code, the
    // lengths, tables and workspace in L2 while the pages stream through.
    const uint64_t kv_policy = l2_policy_evict_first();
    LoadWindow lw{wk, wk.pf, 0, 0, 0, -1};
    if (!wk.done) window_fill(lw, a, P);
    // Half-stages [0, n_issued) have been issued (the live pages of a share
    // form a prefix); after a wait gives up at half-stage x_stop, no more are
    // issued and [x_stop, n_issued) may still be in flight.
    bool timed_out = false;
    int n_issued = 0, x_stop = 0;
    if (a.debug_timeout) {
        // Testing: a wait that runs out before any copy is issued (on a barrier
        // nothing targets, with no time allowed) takes the timeout path below.
        __syncthreads();  // s_never is initialised
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&s_never, 0, 0))) {
            timed_out = true;
            if (lane == 0) flag(a.dev_status, PA_DEV_TIMEOUT);
        }
    }
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
        n_issued = hx + 1;
        if (lane == 0) {
            const int slot = hx % NH;
            const bool ok = pg >= 0 && pg < a.num_pages;
            if (!ok && pg != kDeadPage && (hx & 1) == 0) flag(a.dev_status, PA_DEV_BAD_PAGE);
            my_page[slot] = ok ? pg : -1;
            mbar_arrive_expect_tx(&my_full[slot], ok ? kTile : 0);
            if (ok) {
                uint8_t* dst = my_tiles + size_t(slot) * kTile;
                tma_load_5d_hint(dst, (hx & 1) ? &tmV : &tmK, &my_full[slot], 0, 0, 0, unit_head(a, g), pg,
                                 kv_policy);
            }
        }
        __syncwarp();
    };
    if (!wk.done && !timed_out)
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
    // B fragments of Q^T for unit (b, g): column n = nt*8 + g4 (0 past G)
    auto load_q = [&](uint32_t (&dst)[NT][kKs][2], int b, int g) {
        const int Gu = unit_cols(a, g);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + g4;
            const long long off = row_off<D>(a, b, g, h < Gu ? h : 0);
            const bool in = h < Gu && PA_IN(off / D, a.q_rows, a.dev_status);
            const uint32_t* row = reinterpret_cast<const uint32_t*>(static_cast<const T*>(a.q) + off);
#pragma unroll
            for (int ks = 0; ks < kKs; ++ks) {
                dst[nt][ks][0] = in ? __ldg(row + 8 * ks + t4) : 0u;
                dst[nt][ks][1] = in ? __ldg(row + 8 * ks + 4 + t4) : 0u;
            }
        }
    };
    if (!wk.done) load_q(qn, wk.b, wk.g);
    // Causal lag of the columns this lane holds (heads nt*8 + 2*t4 + j): row t
    // of T sees keys [0, L - (T - 1 - t)).  Padding columns take no lag.  Set
    // per unit (its row block).
    int lag[NT][2];
    int x = 0;  // half-stage number
    // CTA merge (one q-head column tile): the share's first piece, when it is
    // not whole and other units follow, waits here; its last non-whole piece
    // stays in o / mrun / lrun.
    float of[kKs][4], mf[2], lf[2];
    int first_unit = -1, first_inside = 0, last_unit = -1, last_inside = 0;
    float mrun[NT][2], lrun[NT][2];

    while (!wk.done) {
        const int L = __ldg(a.context_lens + wk.b);
        const int Gu = unit_cols(a, wk.g);  // this unit's columns
        {
            const int r0u = unit_row0(a, wk.g);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = nt * 8 + 2 * t4 + j;
                    lag[nt][j] = c < Gu ? a.T - 1 - (r0u + c / a.Gq) : 0;
                }
        }
        const int fp = first_page(a, L, P);  // page i of the unit is page fp + i of the sequence
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
            const int rem = L - (fp + i) * P;  // keys of this page and after it
            const int ntok = min(P, rem);
            // ---- K tile: S^T = K Q^T, masked, online softmax
            bool ok = !timed_out;
            // every lane waits (each needs the barrier's ordering); one outcome per warp
            if (ok && !__all_sync(0xffffffffu, mbar_wait_ns(&my_full[x % NH], (x / NH) & 1, kWaitNs))) {
                timed_out = true;
                x_stop = x;
                ok = false;
                if (lane == 0) flag(a.dev_status, PA_DEV_TIMEOUT);
            }
            const bool valid = ok && my_page[x % NH] >= 0;
            const bool app = a.k_new != nullptr && i == wk.pb - 1;  // the unit's last page holds row L - 1
            if (valid && app)
                append_row<D, P>(my_tiles + size_t(x % NH) * kTile, a.k_new, a.k_cache, a, wk.b, unit_head(a, wk.g),
                                 my_page[x % NH], ntok - 1);
            if (valid) {
                const uint32_t kb = smem_u32(my_tiles + size_t(x % NH) * kTile);
                float s2[kMt][NT][4];  // one column tile: odd k-steps in a second accumulator (shorter chains)
#pragma unroll
                for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[mt][nt][e] = s2[mt][nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kKs; ++ks) {
#pragma unroll
                    for (int mt = 0; mt < kMt; ++mt) {
                        uint32_t ka[4];
                        ldsm_x4(kb + mt * 2048 + offK[ks], ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_16816<kBf>((NT == 1 && (ks & 1)) ? s2[mt][nt] : sc[mt][nt], ka, qb[nt][ks][0],
                                           qb[nt][ks][1]);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[mt][nt][e] += s2[mt][nt][e];
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
                            const int hi = rem - lag[nt][e & 1];  // keys [hi - window, hi) are visible
                            const bool vis = tok < hi && (a.window <= 0 || tok >= hi - a.window);
                            const float v = vis ? sc[mt][nt][e] * a.scale_log2 : -INFINITY;
                            sc[mt][nt][e] = v;
                            mx[nt][e & 1] = fmaxf(mx[nt][e & 1], v);
                        }
                bool same = true;
                float al[NT][2], msf[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float v = mx[nt][j];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        const float mn = fmaxf(mrun[nt][j], v);
                        // no visible key yet (a row of several whose keys end
                        // before this page): offset 0 keeps every weight 0
                        msf[nt][j] = mn == -INFINITY ? 0.f : mn;
                        al[nt][j] = ex2(mrun[nt][j] - msf[nt][j]);  // m = -inf -> 0
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
                            sc[mt][nt][e] = ex2(sc[mt][nt][e] - msf[nt][e & 1]);
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
            if (ok && !__all_sync(0xffffffffu, mbar_wait_ns(&my_full[x % NH], (x / NH) & 1, kWaitNs))) {
                timed_out = true;
                x_stop = x;
                ok = false;
                if (lane == 0) flag(a.dev_status, PA_DEV_TIMEOUT);
            }
            if (valid && ok) {
                uint8_t* vt = my_tiles + size_t(x % NH) * kTile;
                if (app)
                    append_row<D, P>(vt, a.v_new, a.v_cache, a, wk.b, unit_head(a, wk.g), my_page[x % NH], ntok - 1);
                // keys before every row's window in the first window page are
                // never read: zero their V rows (0 * NaN would poison P V)
                const int vlo = a.window > 0 && i == 0 ? L - a.T + a.t0 - a.window + 1 - fp * P : 0;
                if (vlo > 0) {
                    for (int y = lane; y < vlo * kHalves * 8; y += 32) {
                        const int rowi = y / (kHalves * 8), rr = y % (kHalves * 8);
                        *reinterpret_cast<uint4*>(vt + (rr >> 3) * (P * 128) + rowi * 128 + (rr & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
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
        const int unit = wk.b * a.Hv + wk.g;
        if (whole) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int h = nt * 8 + 2 * t4 + j;
                    if (h < Gu && PA_IN(row_off<D>(a, wk.b, wk.g, h) / D, a.out_rows, a.dev_status)) {
                        float* ob = a.out + row_off<D>(a, wk.b, wk.g, h);
                        const float inv = lrun[nt][j] > 0.f ? 1.f / lrun[nt][j] : 0.f;
#pragma unroll
                        for (int dt = 0; dt < kKs; ++dt) {
                            ob[16 * dt + g4] = o[dt][nt][j] * inv;
                            ob[16 * dt + g4 + 8] = o[dt][nt][2 + j] * inv;
                        }
                    }
                }
        } else if (cta_merge) {
            if constexpr (kCtaMerge) {
                const long long p0 = wk.start + a.unit_cost;  // the unit's pages: [p0, p0 + pb)
                const int inside = p0 >= cta_s && p0 + wk.pb <= cta_e;
                if (!nx.done) {  // the share's first piece; later units follow
                    first_unit = unit;
                    first_inside = inside;
                    if (lane == 0) {  // where the unit's pages sit (the counted single launch)
                        s_p0[warp][0] = p0;
                        s_pb[warp][0] = wk.pb;
                    }
#pragma unroll
                    for (int dt = 0; dt < kKs; ++dt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) of[dt][e] = o[dt][0][e];
                    mf[0] = mrun[0][0];
                    mf[1] = mrun[0][1];
                    lf[0] = lrun[0][0];
                    lf[1] = lrun[0][1];
                } else {
                    last_unit = unit;
                    last_inside = inside;
                    if (lane == 0) {
                        s_p0[warp][1] = p0;
                        s_pb[warp][1] = wk.pb;
                    }
                }
            }
        } else {
            const long long slot = PA_IN(part + unit, a.ws_slots, a.dev_status) ? part + unit : -1;
            float* accp = a.ws_acc + slot * G * D;
            float* ml = a.ws_ml + slot * G * 2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int h = nt * 8 + 2 * t4 + j;
                    if (h < G && slot >= 0) {
#pragma unroll
                        for (int dt = 0; dt < kKs; ++dt) {
                            accp[h * D + 16 * dt + g4] = o[dt][nt][j];
                            accp[h * D + 16 * dt + g4 + 8] = o[dt][nt][2 + j];
                        }
                        if (g4 == 0) *reinterpret_cast<float2*>(ml + h * 2) = make_float2(mrun[nt][j], lrun[nt][j]);
                    }
                }
        }
        if (nx.done) break;  // o / mrun / lrun keep the last piece
        wk = nx;
    }
    // A wait that gave up leaves half-stages [x_stop, n_issued) (at most NH)
    // possibly in flight: wait for each of them, bounded by the global timer,
    // before the ring is reused for the merge or the CTA exits.  (The results
    // are already void, PA_DEV_TIMEOUT being set; the merge and the unit
    // counters still run so that every counter is left at zero.)
    if (timed_out)
        for (int y = x_stop; y < n_issued; ++y) mbar_wait_ns(&my_full[y % NH], (y / NH) & 1, kWaitNs);
    __syncwarp();
    if (kCtaMerge && cta_merge) {
        // Stage the non-whole pieces in this warp's own ring (its copies are
        // all consumed): piece k is [G][D + 4] accumulators (the pad puts the
        // 8 x 4 lanes of one store in 32 distinct banks) then [G] (m, l) pairs.
        constexpr int kRow = D + 4;
        const int pstride = (G * kRow + 2 * G + 3) & ~3;  // pieces stay 16-byte aligned
        auto stage = [&](int k, const float (&src)[kKs][4], const float (&m)[2], const float (&l)[2]) {
            float* pc = reinterpret_cast<float*>(my_tiles) + k * pstride;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = 2 * t4 + j;
                if (h < G) {
#pragma unroll
                    for (int dt = 0; dt < kKs; ++dt) {
                        pc[h * kRow + 16 * dt + g4] = src[dt][j];
                        pc[h * kRow + 16 * dt + g4 + 8] = src[dt][2 + j];
                    }
                    if (g4 == 0) {
                        pc[G * kRow + 2 * h] = m[j];
                        pc[G * kRow + 2 * h + 1] = l[j];
                    }
                }
            }
        };
        if (first_unit >= 0) stage(0, of, mf, lf);
        if (last_unit >= 0) {
            float ol[kKs][4], ml_[2] = {mrun[0][0], mrun[0][1]}, ll[2] = {lrun[0][0], lrun[0][1]};
#pragma unroll
            for (int dt = 0; dt < kKs; ++dt)
#pragma unroll
                for (int e = 0; e < 4; ++e) ol[dt][e] = o[dt][0][e];
            stage(1, ol, ml_, ll);
        }
        if (lane == 0) {
            s_unit[warp][0] = first_unit;
            s_inside[warp][0] = first_inside;
            s_unit[warp][1] = last_unit;
            s_inside[warp][1] = last_inside;
        }
        __syncthreads();
        // Merge, unit by unit in warp order, the pieces that warps of this CTA
        // share; a unit whose pages all lie in this CTA's share is finished
        // here, the others leave one piece for the combine (slot CTA + unit).
        // Every warp reads the 16 entry descriptors (lane f and f + 16 hold
        // entry f) and finds, with ballots, where each unit's entries start and
        // which entries hold it.  The code stays short: it runs once per CTA
        // and launch, so its instructions are fetched cold.
        const int f = lane & (2 * kCW - 1);
        const int su = s_unit[f >> 1][f & 1];
        const uint32_t vmask = __ballot_sync(0xffffffffu, su >= 0) & 0xffffu;
        const uint32_t lower = vmask & ((1u << f) - 1u);
        const int pu = __shfl_sync(0xffffffffu, su, lower ? 31 - __clz(lower) : 0);
        const uint32_t starts = __ballot_sync(0xffffffffu, su >= 0 && (lower == 0 || pu != su)) & 0xffffu;
        auto piece = [&](int ff) {
            return reinterpret_cast<const float*>(base + size_t(ff >> 1) * NH * kTile) + (ff & 1) * pstride;
        };
        int k = 0;  // run index: the counted single launch finishes the runs that leave the CTA
        for (uint32_t sm = starts; sm; sm &= sm - 1, ++k) {
            const int e = __ffs(sm) - 1;
            const int u = __shfl_sync(0xffffffffu, su, e);
            const uint32_t emask = __ballot_sync(0xffffffffu, su == u) & 0xffffu;
            const bool inside = s_inside[e >> 1][e & 1] != 0;
            if (threadIdx.x == 0) s_run[k] = make_int4(u, int(emask), inside, e);
            const int ub = u / a.Hv, ug = u % a.Hv;
            // Weights: warp w takes heads 2w and 2w + 1, one lane per entry;
            // maxima and denominators by fixed 16-lane shuffle trees.
            if (2 * warp < G) {
                const int h = 2 * warp + (lane >> 4);
                const bool mine = h < G && ((emask >> f) & 1u);
                const float mm = mine ? piece(f)[G * kRow + 2 * h] : -INFINITY;
                const float ll = mine ? piece(f)[G * kRow + 2 * h + 1] : 0.f;
                float M = mm;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                const float w = mm != -INFINITY ? ex2(mm - M) : 0.f;
                float den = w * ll;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
                if (h < G) {
                    s_w[h][f] = w;
                    if (f == 0) {
                        s_md[h][0] = M;
                        s_md[h][1] = den;
                    }
                }
            }
            __syncthreads();
            for (int idx = threadIdx.x; idx < G * D / 4; idx += kThreadsV1) {
                const int h = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
                float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t m = emask;
                while (m) {  // two entries a step, in ascending order
                    const int f0 = __ffs(m) - 1;
                    m &= m - 1;
                    const int f1 = m ? __ffs(m) - 1 : f0;
                    const float w0 = s_w[h][f0], w1 = m ? s_w[h][f1] : 0.f;
                    const float4 v0 = *reinterpret_cast<const float4*>(piece(f0) + h * kRow + d4);
                    const float4 v1 = *reinterpret_cast<const float4*>(piece(f1) + h * kRow + d4);
                    if (m) m &= m - 1;
                    num.x = fmaf(w1, v1.x, fmaf(w0, v0.x, num.x));
                    num.y = fmaf(w1, v1.y, fmaf(w0, v0.y, num.y));
                    num.z = fmaf(w1, v1.z, fmaf(w0, v0.z, num.z));
                    num.w = fmaf(w1, v1.w, fmaf(w0, v0.w, num.w));
                }
                const float M = s_md[h][0], den = s_md[h][1];
                if (inside) {
                    const float inv = den > 0.f ? 1.f / den : 0.f;
                    if (h < unit_cols(a, ug) && PA_IN(row_off<D>(a, ub, ug, h) / D, a.out_rows, a.dev_status))
                        *reinterpret_cast<float4*>(a.out + row_off<D>(a, ub, ug, h) + d4) =
                            make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
                } else if (PA_IN((long long)blockIdx.x + u, a.ws_slots, a.dev_status)) {
                    const long long slot = (long long)blockIdx.x + u;
                    *reinterpret_cast<float4*>(a.ws_acc + (slot * G + h) * D + d4) = num;
                    if (d4 == 0) *reinterpret_cast<float2*>(a.ws_ml + (slot * G + h) * 2) = make_float2(M, den);
                }
            }
            __syncthreads();  // s_w / s_md are reused by the next unit
        }
        const int nruns = k;
        if (a.finish) {
            // Every CTA piece of this CTA is written (barrier); one thread per
            // run orders them before counting them on the unit's counter
            // (release), and the CTA whose count completes a unit merges the
            // unit's CTA pieces, read through L2, in ascending CTA order (so
            // the result does not depend on which CTA came last), then zeroes
            // the counter.
            __syncthreads();
            if (threadIdx.x < nruns && !s_run[threadIdx.x].z) {
                const int e = s_run[threadIdx.x].w;
                const long long p0 = s_p0[e >> 1][e & 1];
                long long c0 = ((p0 + 1) * n_cta - 1) / cost;  // CTA owning the unit's first page
                const long long c1 = ((p0 + s_pb[e >> 1][e & 1]) * n_cta - 1) / cost;  // and its last
                if (!PA_IN(c0, kMaxCounters, a.dev_status)) c0 = 0;
                const unsigned seen = atom_add_acq_rel_gpu(a.ws_cnt + c0, 1u);
                if (seen == unsigned(c1 - c0)) {
                    s_fin[threadIdx.x] = make_int2(s_run[threadIdx.x].x, int(c0));
                    s_fnp[threadIdx.x] = int(c1 - c0 + 1);
                }
            }
            __syncthreads();
            for (int r = 0; r < nruns; ++r) {
                const int u = s_fin[r].x;
                if (u < 0) continue;
                finish_unit<D>(a, u, s_fin[r].y, s_fnp[r]);
                if (threadIdx.x == 0) a.ws_cnt[s_fin[r].y] = 0u;
            }
        }
    }
    if (kCtaMerge && a.finish) {
        // Sequences with an invalid length have no work units: their rows are
        // written as zeros here (the combine kernel does this otherwise).
        for (long long b = blockIdx.x; b < a.B; b += n_cta) {
            if (seq_pages(a, int(b), P) > 0) continue;
            if (threadIdx.x == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
            const int per_row = a.Hq * D / 4;
            for (int i = threadIdx.x; i < a.Tl * per_row; i += kThreadsV1) {
                const int t = i / per_row;
                if (PA_IN((b * a.T + a.t0 + t) * a.Hq, a.out_rows, a.dev_status))
                reinterpret_cast<float4*>(a.out + ((b * a.T + a.t0 + t) * a.Hq) * D)[i - t * per_row] =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
}

// Merges the pieces of units that span several parts: one CTA per (sequence,
// row, q head), one thread per output dim (head_dim 256: see below).  The CTA locates its pieces from the
// lengths alone (a lane-parallel prefix over the sequences) before it waits
// for the partial kernel through programmatic dependent launch; after the
// wait, the (m, l) pairs of up to 28 pieces (one per lane) and their
// accumulators (one per thread and piece) are loaded together, so a merge
// costs about one L2 round trip.  Maxima and denominators are reduced by
// fixed shuffle trees and the accumulators are summed in ascending part
// order, so the result does not depend on timing.  At most 64 registers a
// thread (1024/D CTAs an SM), so the CTAs that start while the partial kernel
// runs fit beside its 256 x 224-register CTA.
//
// Head_dim 256 (warps leave ~150 pieces per q head): DS CTAs (grid y) share
// an item's dims, and in each, NG groups of D / DS threads merge contiguous
// runs of the pieces with their loads in flight together; group 0 merges
// the groups' results in group order through shared memory.  A CTA keeps to
// 128 threads of 64 registers: one then fits beside a partial-kernel CTA.
template <int D, int NG, int DS>
__global__ void __launch_bounds__(D / DS * NG, 1024 / (D / DS * NG)) combine_v1(const V1Params a, int P) {
    constexpr int kBatch = 28;   // pieces loaded together
    constexpr int kDc = D / DS;  // dims of this CTA
    pdl_launch_dependents();     // the next kernel may start its own set-up
    const int lane = threadIdx.x & 31, dl = threadIdx.x % kDc, grp = threadIdx.x / kDc;
    const int d = int(blockIdx.y) * kDc + dl;
    const int Tb = a.Tl;           // rows of this launch
    const int item = blockIdx.x;  // (b * Tb + t) * Hq + q head
    const int b = item / (Tb * a.Hq), rt = item % (Tb * a.Hq), t = rt / a.Hq, hq = rt % a.Hq;
    const int k = t / a.rb;                             // row block
    const int g = (hq / a.Gq) * a.NB + k;               // unit within the sequence
    const int r = (t - k * a.rb) * a.Gq + hq % a.Gq, h = hq;  // r: the unit's column
    const int unit = b * a.Hv + g;
    const int W = a.unit_cost;
    long long T = 0, pre = 0;
    for (int x = lane; x < a.B; x += 32) {
        const int pg = part_pages(a, x, P);
        const long long c = pg > 0 ? (long long)a.Hv * (pg + W) : 0;
        T += c;
        if (x < b) pre += c;
    }
    T = warp_sum_ll(T);
    pre = warp_sum_ll(pre);
    const int pp = part_pages(a, b, P);  // the unit's pages in the partition
    const int pb = seq_pages(a, b, P);   // 0: an invalid length
    const long long nc = ctas_in_use(T > 0 ? T : 1, a.n_ctas);
    const bool cta = a.cta_pieces && T <= (long long)kCtaMergeMaxShare * nc;  // as the partial kernel
    const long long n = cta ? nc : nc * warps_in_use(T, nc);  // parts of the piece partition
    long long c0 = 0;
    int np = 0;
    if (pb > 0) {  // the unit's pages sit at cost positions [p0, p0 + pp)
        const long long p0 = pre + (long long)g * (pp + W) + W;
        c0 = ((p0 + 1) * n - 1) / T;  // part v owns [v*T/n, (v+1)*T/n)
        const long long c1 = ((p0 + pp) * n - 1) / T;
        np = c1 > c0 ? int(c1 - c0 + 1) : 0;  // 0: finished inside one part
    }
    pdl_wait_primary();  // the partial kernel's pieces are complete from here on
    const long long orow = ((long long)b * a.T + a.t0 + t) * a.Hq + hq;
    if (!PA_IN(orow, a.out_rows, a.dev_status)) return;
    float* o = a.out + orow * D + d;
    if (pb == 0) {
        if (grp == 0) *o = 0.f;
        if (h == 0 && d == 0) flag(a.dev_status, PA_DEV_BAD_LEN);
        return;
    }
    if (np == 0) return;
    // Parts between c0 and c1 whose share is empty (possible when T < n) wrote
    // nothing: their weight is 0 and their rows are never used.
    const int per = (np + NG - 1) / NG;  // this group's pieces: [lo, hi)
    const int lo = min(np, grp * per), hi = min(np, lo + per);
    float M = -INFINITY, den = 0.f, num = 0.f;
    for (int x0 = lo; x0 < hi; x0 += kBatch) {
        const int cnt = min(kBatch, hi - x0);
        float mj = -INFINITY, lj = 0.f;
        if (lane < cnt) {
            const long long cc = c0 + x0 + lane;
            if ((T >= n || cc * T / n != (cc + 1) * T / n) &&  // T >= n: no share is empty
                PA_IN(cc + unit, a.ws_slots, a.dev_status)) {
                const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + ((cc + unit) * a.G + r) * 2);
                mj = ml.x;
                lj = ml.y;
            }
        }
        const float* accp = a.ws_acc + ((c0 + x0 + unit) * a.G + r) * D + d;
        float v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            v[j] = j < cnt && PA_IN(c0 + x0 + j + unit, a.ws_slots, a.dev_status) ? accp[(long long)j * a.G * D] : 0.f;
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
    if constexpr (NG == 1) {
        *o = den > 0.f ? num / den : 0.f;
    } else {
        __shared__ float s_num[NG][kDc], s_m[NG], s_den[NG];
        s_num[grp][dl] = num;
        if (dl == 0) {
            s_m[grp] = M;
            s_den[grp] = den;
        }
        __syncthreads();
        if (grp != 0) return;
        float Mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < NG; ++k) Mt = fmaxf(Mt, s_m[k]);
        float nn = 0.f, dd = 0.f;
        if (Mt != -INFINITY)
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const float w = s_m[k] == -INFINITY ? 0.f : ex2(s_m[k] - Mt);
                dd = fmaf(w, s_den[k], dd);
                nn = fmaf(w, s_num[k][dl], nn);
            }
        *o = dd > 0.f ? nn / dd : 0.f;
    }
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
// combine CTA (the per-CTA reservation) and the kernel's static shared memory
// have room.
int tile_count(int D, int P) {
    const size_t tile = size_t(P) * D * 2;
    const size_t room = size_t(kSmemLimit) - 1024 - v1_fixed_bytes() - 2048 - 1024;
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
    const size_t dyn = smem_bytes(D, P, a.ntiles);  // a function of (D, P) alone
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // Programmatic dependent launch: the CTAs may start (and set up shared
    // memory) while the previous kernel on the stream finishes; the kernel
    // waits for it before its first global-memory access.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(kThreadsV1);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, k, v, a);
}

template <typename T, int D, int P>
cudaError_t launch_typed(const CUtensorMap& k, const CUtensorMap& v, const V1Params& a, int n_ctas,
                         int phases, cudaStream_t st) {
    if (phases & 1) {
        // one 8-wide column tile of q heads when the group fits, else two
        cudaError_t e;
        if constexpr (D == 256) {  // one column tile only (accumulator registers)
            e = a.G <= 8 ? launch_partial<T, D, P, 1>(k, v, a, n_ctas, st) : cudaErrorInvalidValue;
        } else {
            e = a.G <= 8 ? launch_partial<T, D, P, 1>(k, v, a, n_ctas, st)
                         : launch_partial<T, D, P, 2>(k, v, a, n_ctas, st);
        }
        if (e != cudaSuccess) return e;
    }
    if (!(phases & 2) || a.finish) return cudaSuccess;  // single launch: no combine kernel
    cudaLaunchConfig_t cfg = {};
    // Every combine CTA has 128 threads at most (8,192 registers), so one fits
    // beside a partial-kernel CTA and the next call's partial CTAs find room
    // beside the combine's.  D 256: eight CTAs an item, each with 32 dims and
    // four piece groups of one warp.
    constexpr int kGroups = D == 256 ? 4 : 1;  // piece groups of a combine CTA
    constexpr int kSplit = D == 256 ? 8 : 1;   // CTAs per item, each with D / kSplit dims
    cfg.gridDim = dim3(unsigned(a.B) * unsigned(a.Tl) * unsigned(a.Hq), kSplit);
    cfg.blockDim = dim3(D / kSplit * kGroups);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_v1<D, kGroups, kSplit>, a, P);
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: the arrival counters of the single launch (a fixed block that
// must be zero before a call and is left zero by it), then (m, l) pairs, then
// accumulators, one slot per (part, unit) piece of G columns; Hv units per
// sequence.
struct WsLayout {
    size_t cnt, ml, acc, total;
};
WsLayout ws_layout(int B, int Hv, int G, int D, int n_ctas) {
    const size_t slots = size_t(n_ctas) * kCW + size_t(B) * Hv;
    WsLayout w;
    w.cnt = 0;
    w.ml = w.cnt + size_t(kMaxCounters) * sizeof(unsigned);
    w.acc = w.ml + round256(slots * G * 2 * sizeof(float));
    w.total = w.acc + slots * G * D * sizeof(float);
    return w;
}

}  // namespace

size_t decode_v1_workspace_bytes(int B, int Hkv, int G, int NB, int D, int n_ctas) {
    return ws_layout(B, Hkv * NB, G, D, n_ctas).total;
}


// The kernel parameters of a call (all but the tensor maps).
cudaError_t build_params(const DecodeV1Call& call, V1Params& a) {
    const int D = call.D, P = call.P;
    a.q = call.q;
    a.block_tables = call.block_tables;
    a.context_lens = call.context_lens;
    a.out = call.out;
    const int T = call.rows > 0 ? call.rows : 1;
    const int nr = call.row_count > 0 ? call.row_count : T;  // rows of this launch
    const int rb = call.row_block > 0 && call.row_block < nr ? call.row_block : nr;  // rows of a unit
    const int NB = (nr + rb - 1) / rb;
    const int G = rb * (call.Hq / call.Hkv);  // columns per unit: rows x q heads of a kv head
    if (G > 16 || call.row0 < 0 || call.row0 + nr > T) return cudaErrorInvalidValue;
    const WsLayout wl = ws_layout(call.B, call.Hkv * NB, G, D, call.n_ctas);
    char* ws = static_cast<char*>(call.workspace);
    a.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    a.ws_acc = reinterpret_cast<float*>(ws + wl.acc);
    a.ws_cnt = reinterpret_cast<unsigned*>(ws + wl.cnt);
    a.ws_slots = (long long)call.n_ctas * kCW + (long long)call.B * call.Hkv * NB;
    a.q_rows = a.out_rows = (long long)call.B * T * call.Hq;
    a.dev_status = call.dev_status;
    a.B = call.B;
    a.Hq = call.Hq;
    a.Hkv = call.Hkv;
    a.G = G;
    a.T = T;
    a.t0 = call.row0;
    a.Tl = nr;
    a.rb = rb;
    a.NB = NB;
    a.Hv = call.Hkv * NB;
    a.Gq = call.Hq / call.Hkv;
    a.num_pages = call.num_pages;
    a.max_blocks = call.max_blocks;
    a.max_len = call.max_blocks * P;
    a.scale_log2 = call.scale_log2;
    a.n_ctas = call.n_ctas;
    a.window = call.window;
    a.debug_timeout = call.debug_timeout;
    // Static plan for small calls (no window, no append): every sequence
    // counts max_context_len's pages in the partition when that whole space
    // is a small call (shares of at most kCtaMergeMaxShare cost units).
    {
        const long long pmax = (call.max_context_len + P - 1) / P;
        const bool small = (long long)call.B * a.Hv * (pmax + kUnitCost) <=
                           (long long)kCtaMergeMaxShare * call.n_ctas;
        a.static_pages = call.window == 0 && call.k_new == nullptr && small && pmax > 0 ? int(pmax) : 0;
    }
    a.cta_pieces = G <= 8 && D <= 128;  // as the partial kernel's kCtaMerge
    a.finish = a.cta_pieces && call.phases == 3 && call.single_launch;  // one launch for the whole call
    a.k_new = call.k_new;
    a.v_new = call.v_new;
    a.k_cache = const_cast<void*>(call.k);
    a.v_cache = const_cast<void*>(call.v);
    a.page_stride = call.page_stride;
    a.token_stride = call.token_stride;
    a.head_stride = call.head_stride;
    a.ntiles = tile_count(D, P);
    a.unit_cost = kUnitCost;
    // at least one page tile per warp (head_dim 256 with 32-slot pages has
    // one: its K and V copies then take turns in it)
    if (a.ntiles < kCW || call.n_ctas > kMaxCounters) return cudaErrorInvalidValue;
    return cudaSuccess;
}

int decode_v1_kernels(const DecodeV1Call& call) {
    V1Params a;
    if (build_params(call, a) != cudaSuccess) return -1;
    if (!(call.phases & 1)) return (call.phases & 2) && !a.finish ? 1 : 0;
    return a.finish ? 1 : ((call.phases & 2) ? 2 : 1);
}

cudaError_t launch_decode_v1(const DecodeV1Call& call, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int D = call.D, P = call.P;
    const CUtensorMapDataType dt =
        call.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // The pool as a 5-d tensor (dim within a 64-dim half, slot, half, kv head,
    // page), with each dimension's own stride: the box (64 x P x D/64 x 1 x 1)
    // is one page of one kv head in one copy, and lands in shared memory as
    // D/64 blocks of P rows of 128 bytes (the swizzle span), the layout the
    // ldmatrix offsets assume.
    CUtensorMap mk, mv;
    const cuuint64_t dims[5] = {64, cuuint64_t(P), cuuint64_t(D / 64), cuuint64_t(call.Hkv),
                                cuuint64_t(call.num_pages)};
    const cuuint64_t strides[4] = {cuuint64_t(call.token_stride) * 2, 128, cuuint64_t(call.head_stride) * 2,
                                   cuuint64_t(call.page_stride) * 2};
    const cuuint32_t box[5] = {64, cuuint32_t(P), cuuint32_t(D / 64), 1, 1}, estr[5] = {1, 1, 1, 1, 1};
    if (enc(&mk, dt, 5, const_cast<void*>(call.k), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (enc(&mv, dt, 5, const_cast<void*>(call.v), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    V1Params a;
    cudaError_t pe = build_params(call, a);
    if (pe != cudaSuccess) return pe;
    const bool bf = call.dtype == PA_BF16;
#define PA_V1_CASE(DD, PP)                                                                        \
    if (D == DD && P == PP)                                                                       \
        return bf ? launch_typed<__nv_bfloat16, DD, PP>(mk, mv, a, call.n_ctas, call.phases, st) \
                  : launch_typed<__half, DD, PP>(mk, mv, a, call.n_ctas, call.phases, st);
    PA_V1_CASE(256, 32)
    PA_V1_CASE(256, 16)
    PA_V1_CASE(128, 32)
    PA_V1_CASE(128, 16)
    PA_V1_CASE(64, 32)
    PA_V1_CASE(64, 16)
#undef PA_V1_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pa
