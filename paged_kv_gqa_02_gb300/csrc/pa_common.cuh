// pa_common.cuh -- device helpers shared by the paged GQA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_gqa.h"

namespace pa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxGroup = 16;  // largest Hq / Hkv ratio the kernels accept

// Arguments shared by the attention kernels.  Pointers are device memory;
// strides are in elements of the KV dtype.
struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* cu_q_lens;  // nullptr: decode, one row per sequence
    float* out;                // final output, or nullptr when writing partials
    float* partial_ml;         // [B][Hq][S][2]
    float* partial_acc;        // [B][Hq][S][D]
    uint32_t* dev_status;      // nullable
    int32_t num_seqs, num_q_heads, num_kv_heads, group;
    int32_t num_pages, max_blocks_per_seq;
    int64_t page_stride, token_stride, head_stride;
    float scale_log2;     // scale * log2(e): scores are kept in base-2 units
    int32_t split_tokens; // keys per split (multiple of page_size)
    int32_t num_splits;   // S
    int32_t max_q_len;    // prefill: host bound on rows per sequence
    int32_t total_q;      // rows in q / out
    int32_t rows_per_seq = 0;  // > 1 with cu_q_lens == nullptr: sequence b owns rows b*n .. b*n + n - 1
    // Extents, in elements, for the checked build's range checks
    int64_t q_elems = 0, out_elems = 0, partial_items = 0;
    int32_t debug_timeout = 0;  // 1: the tensor-core prefill gives up before any copy (testing)
};

// ---- element conversions -------------------------------------------------
template <typename T> struct Elt;
template <> struct Elt<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static inline float f(float x) { return x; }
};
template <> struct Elt<__half> {
    static constexpr int kVec = 8;
    __device__ static inline float f(__half x) { return __half2float(x); }
};
template <> struct Elt<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static inline float f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Converts one 16-byte vector of T into floats.
template <typename T>
__device__ inline void vec_to_f32(const uint4& raw, float* dst) {
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < Elt<T>::kVec; ++i) dst[i] = Elt<T>::f(e[i]);
}

// ---- math ------------------------------------------------------------------
// 2^x through the PTX ex2.approx instruction (flush-to-zero; ex2(-inf) = +0).
__device__ inline float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ inline float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ inline float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ inline void flag(uint32_t* status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// Checked builds (PA_CHECKED defined): PA_IN(i, n, st) is true when the
// computed index i lies in [0, n); otherwise it sets PA_DEV_OOB in *st and is
// false, so the guarded access is skipped.  Release builds compile it to
// `true`: the kernels' index arithmetic keeps every access in range by
// construction, and the checked build is how that is tested.
#ifdef PA_CHECKED
__device__ inline bool checked_in(long long i, long long n, uint32_t* status) {
    if (i >= 0 && i < n) return true;
    flag(status, PA_DEV_OOB);
    return false;
}
#define PA_IN(i, n, st) (::pa::checked_in((long long)(i), (long long)(n), (st)))
#else
#define PA_IN(i, n, st) (true)
#endif

}  // namespace pa
