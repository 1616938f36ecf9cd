// pa_kernels.h -- launchers of the CUDA kernels (internal to the library).
#pragma once

#include "pa_common.cuh"

namespace pa {

// v0 tile kernel: decode split partials (a.out == nullptr) or the final
// output (a.out set, single split); grid (S, Hkv, B).
cudaError_t launch_decode_v0(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st);
// v0 tile kernel over packed prefill rows; grid (ceil(max_q_len/4), Hkv, B).
cudaError_t launch_prefill_v0(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st);
// Split combine, grid (Hq, B), D threads; sequence b merges its first
// splits_per_seq[b] splits (all S when NULL).
cudaError_t launch_combine_v0(const float* ml, const float* acc, float* out, int B, int Hq,
                              int S, int D, cudaStream_t st, const int32_t* splits_per_seq = nullptr);

// v1 decode for 16-bit K/V: persistent length-balanced partial kernel (TMA +
// mma.sync) followed by a PDL-launched combine of split units.
struct DecodeV1Call {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* out;
    void* workspace;  // decode_v1_workspace_bytes(...) bytes, 256-byte aligned
    uint32_t* dev_status;
    pa_dtype dtype;
    int B, Hq, Hkv, D, P, num_pages, max_blocks, n_ctas;
    int64_t page_stride, token_stride, head_stride;
    float scale_log2;
    int phases;  // bit 0: partial kernel, bit 1: combine kernel
    int rows = 1;       // query rows per sequence (causal among them)
    int row0 = 0;       // first row this launch handles
    int row_count = 0;  // rows this launch handles (0: all)
    int row_block = 0;  // rows of a unit (0: row_count); row_block x Hq/Hkv <= 16.  The
                        // launch's rows come in blocks of row_block, each block a unit
    int window = 0;     // > 0: each row sees only its last `window` keys
    int single_launch = 0;  // 1: finish split units in the partial kernel (one column tile, D <= 128)
    int max_context_len = 0;  // host bound on every length (sizes the static plan of small calls)
    int debug_timeout = 0;    // 1: every warp's waits give up before any copy is issued (testing)
    // KV append (both nullptr: none): [B][Hkv][D] rows written to row L_b - 1
    // of the cache and attended in place of what it held
    const void* k_new = nullptr;
    const void* v_new = nullptr;
};
// Chunked prefill on the tensor cores (tcgen05): 16-bit Q/K/V, head_dim 128,
// pages of 16 or 32 slots, G = Hq/Hkv <= 16, scale > 0.  One CTA per (row-tile
// pair, kv head, sequence), the pairs of a (sequence, kv head) consecutive.
bool prefill_tc_supported(pa_dtype dt, int D, int P, int G, float scale);
cudaError_t launch_prefill_tc(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st);

// Writes the new token's K/V rows ([B][Hkv][D]) to row L_b - 1 of each
// sequence's last page; sequences with an invalid length or page are skipped.
cudaError_t launch_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens, int B, int Hkv,
                             int D, int P, int elt_bytes, int num_pages, int max_blocks, int64_t page_stride,
                             int64_t token_stride, int64_t head_stride, cudaStream_t st);

// Hq counts q heads times query rows per sequence.
// Workspace of a launch whose units have G columns, NB row blocks per kv head;
// its first PA_DECODE_COUNTER_BYTES hold the single launch's arrival counters.
size_t decode_v1_workspace_bytes(int B, int Hkv, int G, int NB, int D, int n_ctas);
cudaError_t launch_decode_v1(const DecodeV1Call& call, cudaStream_t st);
// Kernels launch_decode_v1 would launch for this call (1 or 2; -1: invalid).
int decode_v1_kernels(const DecodeV1Call& call);

}  // namespace pa
