/*
 * paged_gqa.h -- C ABI of libpaged_gqa.so: attention over a paged KV cache
 * with grouped-query heads, for NVIDIA GB300 (sm_103a).
 *
 * The operation (crucible paged attention results: the reference kernel,
 * the K/V pool layout and the GQA mapping paragraphs; crucible README,
 * "Layout, and why it was nearly free" and "Prefill scheduling"):
 *
 *   for each sequence s, query row r in [0, T_s), q head h:
 *     g     = h / (num_q_heads / num_kv_heads)           (GQA mapping)
 *     start = L_s - T_s ; end = start + r                (causal bound)
 *     for keys j in [0, end]:
 *       page  = block_tables[s][j / page_size]; slot = j % page_size
 *       k_j   = k_cache[page][slot][g][:], v_j likewise  (through strides)
 *       sigma_j = scale * dot(q[s,r,h,:], k_j)
 *     out[s,r,h,:] = sum_j exp(sigma_j - max sigma) v_j / sum_j exp(sigma_j - max sigma)
 *
 * L_s = context_lens[s] counts the cached history plus this call's T_s rows
 * (their K/V must already be in the pages).  Decode is T_s = 1.
 *
 * Conventions for every entry point:
 *  - Ownership: every pointer argument is device memory owned by the caller
 *    (except `const pa_params*`, which is host memory read during the call).
 *    The library allocates nothing and keeps no per-call state; the only
 *    global memory it uses besides the arguments is the caller's workspace
 *    (one exception: pa_decode_noalloc keeps its split partials in a static
 *    device array of PA_NOALLOC_SCRATCH_BYTES inside the library).
 *  - Asynchrony: calls enqueue work on `stream` and return.  PA_OK means the
 *    arguments passed host validation and the kernels were launched.
 *    Host-detectable errors return before anything is launched.
 *  - Device-detected metadata errors (a block-table entry outside
 *    [0, num_pages), a context length outside [T_s, max_blocks_per_seq *
 *    page_size]) never form an out-of-range address: the affected keys are
 *    skipped, rows with no valid key are written as zeros, and the bits
 *    below are OR-ed into *dev_status when it is non-NULL.  The caller zeroes
 *    dev_status before the call if it wants a fresh reading.
 *  - Graph capture: grid sizes depend only on host-side pa_params fields,
 *    never on device-resident lengths, so calls can be captured in a CUDA
 *    graph and replayed with new lengths and tables.
 *  - Determinism: no value path uses atomics, so a given device returns
 *    bit-identical results for identical inputs on every run.  With
 *    deterministic = 1 the split-KV partition is also independent of the
 *    device (a function of pa_params alone).
 *  - Supported: head_dim in {64, 128} everywhere, and 256 for pa_decode and
 *    pa_decode_append with 16-bit K/V, automatic splits and at most 8 MMA
 *    columns (query rows x Hq/Hkv) per block (PA_ERR_UNSUPPORTED otherwise);
 *    page_size in {16, 32};
 *    num_q_heads % num_kv_heads == 0 with a ratio of at most 16;
 *    q_dtype == kv_dtype in {PA_F32, PA_F16, PA_BF16}; out_dtype = PA_F32;
 *    q, k_cache, v_cache and out 16-byte aligned; head_dim contiguous and
 *    the three cache strides multiples of 16 bytes.
 */
#ifndef PAGED_GQA_H
#define PAGED_GQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pa_stream_t;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* pa_params.decode_form */
enum { PA_FORM_AUTO = 0, PA_FORM_PAIR = 1, PA_FORM_COUNTED = 2 };

typedef enum {
    PA_OK = 0,
    PA_ERR_NULL = 1,        /* a required pointer is NULL                  */
    PA_ERR_SHAPE = 2,       /* inconsistent sizes                           */
    PA_ERR_DTYPE = 3,       /* unknown dtype code                           */
    PA_ERR_ALIGN = 4,       /* pointer or stride not 16-byte aligned        */
    PA_ERR_WORKSPACE = 5,   /* workspace smaller than the *_workspace_size  */
    PA_ERR_UNSUPPORTED = 6, /* valid but not implemented (head_dim, ...)    */
    PA_ERR_CUDA = 7         /* a CUDA runtime call failed                   */
} pa_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define PA_DEV_BAD_PAGE 1u /* a block-table entry outside [0, num_pages) */
#define PA_DEV_BAD_LEN 2u  /* context_len < T_s or > max_blocks_per_seq * page_size */
#define PA_DEV_TIMEOUT 4u  /* a bounded device wait gave up */
/* Library built with PA_CHECKED defined only: a computed global index left
 * its buffer (block table, lengths, q, out, workspace); the access was
 * skipped.  A release build never sets it. */
#define PA_DEV_OOB 8u

typedef struct {
    int32_t num_seqs;           /* B                                           */
    int32_t num_q_heads;        /* Hq                                          */
    int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0, Hq / Hkv <= 16           */
    int32_t head_dim;           /* D: 64 or 128                                */
    int32_t page_size;          /* P: 16 or 32 tokens per page                 */
    int32_t num_pages;          /* pages in the pool (valid table entries)     */
    int32_t max_blocks_per_seq; /* row stride of block_tables                  */
    int32_t max_context_len;    /* host upper bound on every context_lens[s];
                                   sizes the split plan and the workspace       */
    int64_t page_stride;        /* elements between pages; 0 = P*Hkv*D          */
    int64_t token_stride;       /* elements between slots; 0 = Hkv*D            */
    int64_t head_stride;        /* elements between kv heads; 0 = D             */
    float scale;                /* applied to q.k (typically 1/sqrt(D))        */
    pa_dtype q_dtype;           /* dtype of q                                  */
    pa_dtype kv_dtype;          /* dtype of k_cache / v_cache (== q_dtype)      */
    pa_dtype out_dtype;         /* PA_F32                                      */
    int32_t deterministic;      /* 1: split plan from pa_params alone           */
    int32_t num_splits;         /* decode: 0 = automatic, else requested count  */
    int32_t decode_phases;      /* pa_decode: 0 = the whole call (one kernel
                                   when the call takes the single-launch form
                                   below); 1 = partial step only; 2 = combine
                                   step only (after a phase-1 call on the same
                                   workspace, to put other work between the two
                                   or time them).  1 then 2 is the two-kernel
                                   form: equal to the whole call within the
                                   decode tolerances (bit for bit where the
                                   call has no single-launch form)             */
    int32_t decode_q_rows;      /* pa_decode: query rows per sequence, 0 or 1 =
                                   one; up to 16 (speculative / multi-token
                                   decode).  q and out are then [B][rows][Hq][D]
                                   and row t of a sequence of length L sees keys
                                   [0, L - rows + t] (causal among the rows, as
                                   in chunked prefill; crucible README, "Prefill
                                   scheduling").  L < rows is an invalid length.
                                   16-bit K/V with automatic splits run on the
                                   split-KV kernel with the rows as extra MMA
                                   columns, in blocks of 16 / (Hq/Hkv) rows (8 /
                                   (Hq/Hkv) at head_dim 256), each block its own
                                   work unit of one launch; fp32 K/V
                                   take the CUDA-core pass over tiles of 4 rows
                                   x the automatic key splits, then the combine
                                   per (row, q head); num_splits must be 0.
                                   Not with pa_decode_partial or
                                   pa_decode_append.                             */
    int32_t sliding_window;     /* 0: none.  W > 0: a row whose causal end is
                                   key e attends only keys e - W + 1 ..= e, its
                                   last W keys (vllm.cpp PR #383 names a
                                   windowed decode instantiation; this is the
                                   plain reading).  Keys before every row's
                                   window are never read.  pa_decode and
                                   pa_decode_append with 16-bit K/V and
                                   automatic splits only; otherwise
                                   PA_ERR_UNSUPPORTED.                            */
    int32_t decode_form;        /* pa_decode / pa_decode_append with 16-bit K/V,
                                   automatic splits, head_dim <= 128 and rows x
                                   Hq/Hkv <= 8 (see pa_decode):
                                   PA_FORM_AUTO (0, default): the library's
                                   choice, today the partial + combine pair;
                                   PA_FORM_PAIR (1): the pair; PA_FORM_COUNTED
                                   (2): one kernel whose last CTA per unit
                                   merges its pieces.  Other calls ignore it.   */
    int32_t debug_timeout;      /* testing only, 0 otherwise.  1: every wait of
                                   the split-KV decode kernel and of the tensor-
                                   core prefill kernel gives up at once, before
                                   any copy is issued (each first waits with no
                                   time allowed on a barrier that no copy
                                   targets), so the kernels take their
                                   timeout path: PA_DEV_TIMEOUT is set, nothing
                                   is read from the cache and the results are
                                   void (zeros).  Shows that a wait that runs
                                   out leaves the context usable.               */
} pa_params;

/* Fills *p with defaults: contiguous strides, PA_F32 out, automatic splits,
 * deterministic = 1; sizes and dtypes zero.  Returns p. */
pa_params *pa_params_init(pa_params *p);

/* Human-readable name of a status code (static storage). */
const char *pa_status_string(pa_status s);

/* ------------------------------------------------------------------ decode
 * One query row per sequence: q and out are [B][Hq][D] (row-major), q in
 * q_dtype, out in f32.  block_tables is [B][max_blocks_per_seq] int32,
 * context_lens is [B] int32, both on the device.
 *
 * Split-KV (crucible README "Split-position attention"; minfer doc 71,
 * Excerpts F and G): the keys of each (sequence, kv head) are cut into
 * splits of `split_tokens` keys (a multiple of page_size).  The plan is
 * fixed by pa_params (never by device lengths), so the grid is constant.
 */

/* Split plan: *num_splits = S (splits per sequence at max_context_len) and
 * *split_tokens = keys per split.  Either output may be NULL. */
pa_status pa_decode_plan(const pa_params *p, int32_t *num_splits, int32_t *split_tokens);

/* Kernels one pa_decode call (with_append = 0) or pa_decode_append call
 * (with_append = 1) launches for these parameters: 1 for the counted single
 * launch and single-split calls, 2 for the partial + combine pair, 3 when
 * the append needs its scatter kernel, and so on; -1 for invalid or
 * unsupported parameters.  For callers that budget graph nodes. */
int32_t pa_decode_kernels(const pa_params *p, int32_t with_append);

/* Bytes of workspace pa_decode needs for these parameters (0 on the fixed
 * split path when the plan has a single split).  Returns 0 for invalid
 * parameters. */
size_t pa_decode_workspace_size(const pa_params *p);

/* Decode attention: the split partials and their combine.
 * workspace: device memory of at least pa_decode_workspace_size(p) bytes,
 * 256-byte aligned.  Its first PA_DECODE_COUNTER_BYTES bytes hold arrival
 * counters: they must be zero before the first pa_decode or
 * pa_decode_append call that uses the buffer (zero the whole buffer once
 * after allocating it, e.g. with cudaMemsetAsync), and every call leaves
 * them zero, whatever its parameters, so a buffer is zeroed once.  The
 * other bytes are scratch: contents ignored.  dev_status may be NULL.
 *
 * With num_splits = 0 and 16-bit K/V the partition is length-balanced: one
 * persistent CTA per SM (a fixed 152 when deterministic = 1, the device's
 * SM count otherwise; 8 warps each) takes equal contiguous shares of the
 * ordered (sequence, kv head [, row block], page) list, and its warps split
 * the share the same way (fewer warps for small calls when the group needs
 * two MMA column tiles or head_dim is 256); units that fall inside one
 * share are finished there.  The pieces of the others are merged in
 * ascending share order:
 *  - by a second kernel, launched with programmatic dependent launch so that
 *    its CTAs are resident and have located their pieces when the partial
 *    kernel ends (PA_FORM_AUTO and PA_FORM_PAIR);
 *  - PA_FORM_COUNTED, head_dim <= 128 and rows x Hq/Hkv <= 8: in the partial
 *    kernel itself, each CTA merges its warps' pieces and the last CTA to
 *    leave a piece of a unit (counted on a workspace counter with an
 *    acquire-release atomic) merges the unit's CTA pieces.  One kernel; on
 *    GB300 it takes longer than the pair, because the count and the
 *    finishing CTA's reads sit on the critical path after the slowest CTA.
 * Otherwise the fixed split plan of pa_decode_plan is used (the
 * pa_decode_partial + pa_combine pair). */
#define PA_DECODE_COUNTER_BYTES 4096u

pa_status pa_decode(const pa_params *p, const void *q, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables,
                    const int32_t *context_lens, float *out, void *workspace,
                    size_t workspace_bytes, uint32_t *dev_status, pa_stream_t stream);

/* Decode with the new token's K/V appended in the same pass.  The pages
 * scatter each new token's K and V into the paged pool before attention on
 * the same stream (crucible paged attention results, the layer walk-through;
 * crucible README, "Layout, and why it was nearly free": decode's K/V write
 * goes through the page table).  For each sequence b with a valid length L_b
 * (which counts the new token) and a valid page
 * pg = block_tables[b][(L_b - 1) / page_size], rows k_new[b][g][:] and
 * v_new[b][g][:] of every kv head g are written to slot (L_b - 1) % page_size
 * of page pg of k_cache / v_cache; then out is pa_decode's over keys
 * [0, L_b), the new token included.  Whatever the slot held before is
 * neither read nor used.
 *   k_new, v_new: [B][Hkv][D] in kv_dtype, contiguous, 16-byte aligned,
 *                 device memory owned by the caller.
 *   k_cache, v_cache: written at those slots only (caller-owned).
 * Other arguments, the workspace, asynchrony and errors are as pa_decode's.
 * With 16-bit K/V and automatic splits the write happens inside the
 * attention kernel: the warp that copies a sequence's last page into shared
 * memory replaces the row there and stores it to the cache.  Otherwise a
 * scatter kernel writes the rows before the attention.  The slot must not
 * be shared with another sequence of the same call. */
pa_status pa_decode_append(const pa_params *p, const void *q, const void *k_new,
                           const void *v_new, void *k_cache, void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           float *out, void *workspace, size_t workspace_bytes,
                           uint32_t *dev_status, pa_stream_t stream);

/* The partial step on its own.  For each sequence b, q head h and split i
 * in [0, num_splits) (num_splits from pa_decode_plan) it writes, with
 * idx = (b*Hq + h)*num_splits + i:
 *   partial_ml[2*idx]     = m: the largest scaled score of the split times
 *                           log2(e) (base-2 units), -inf for an empty split
 *   partial_ml[2*idx + 1] = l: sum over the split of 2^(score*log2e - m)
 *   partial_acc[idx*D ..] = sum over the split of 2^(score*log2e - m) v_j
 *                           (not written for an empty split)
 * partial_ml is [B][Hq][S][2] f32, partial_acc is [B][Hq][S][D] f32. */
pa_status pa_decode_partial(const pa_params *p, const void *q, const void *k_cache,
                            const void *v_cache, const int32_t *block_tables,
                            const int32_t *context_lens, float *partial_ml,
                            float *partial_acc, int32_t num_splits,
                            uint32_t *dev_status, pa_stream_t stream);

/* Combine (crucible README "Split-position attention": rescale each split
 * by exp(m_i - m_max) and merge; minfer doc 71 Excerpt F: idle splits write
 * m = -inf and get weight zero).  partial_ml is [B][Hq][max_splits][2] and
 * partial_acc [B][Hq][max_splits][D] (the layout pa_decode_partial writes).
 * For each (b, h), over splits i < S_b in ascending order:
 *   M = max_i m_i;  w_i = 2^(m_i - M) (0 when m_i = -inf);
 *   out[b][h][:] = sum_i w_i acc_i / sum_i w_i l_i,  or 0 when every m_i = -inf.
 * S_b = splits_per_seq[b] clamped to [0, max_splits] when splits_per_seq
 * (device memory, [B] int32) is non-NULL, else max_splits; splits at or
 * past S_b are never read (S_b = 0 writes zeros).
 * Uses p->num_seqs, num_q_heads, head_dim; out is [B][Hq][D] f32.
 * partial_acc and out 16-byte aligned, partial_ml 8-byte aligned. */
pa_status pa_combine(const pa_params *p, const float *partial_ml, const float *partial_acc,
                     int32_t max_splits, const int32_t *splits_per_seq, float *out,
                     pa_stream_t stream);

/* Decode without a workspace argument (the pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory at call
 * time, such as an engine plugin whose host owns all device buffers, a
 * serving loop that forbids allocation after start-up, or a process whose
 * caching allocator already holds the free memory).
 *
 * It runs the fixed split plan of pa_decode_plan (pa_decode_partial, then
 * pa_combine: the path pa_decode takes when num_splits is set), keeping the
 * split partials in a static device array of PA_NOALLOC_SCRATCH_BYTES
 * inside the library.  Its result equals pa_decode's within the decode
 * tolerances; where pa_decode takes the same plan (fp32 K/V with several
 * splits, or num_splits > 0) both run the same kernels.  Several query rows,
 * sliding windows and head_dim 256 return PA_ERR_UNSUPPORTED, as for
 * pa_decode_partial.  Every GPU that loads the
 * library holds that array until the process exits.  It allocates nothing
 * and calls no allocating routine.
 *  - Limit: when the plan's partials (B * Hq * S * (D + 2) floats, each part
 *    rounded up to 256 bytes) exceed PA_NOALLOC_SCRATCH_BYTES it returns
 *    PA_ERR_WORKSPACE and launches nothing; use pa_decode with a workspace
 *    or request fewer splits (pa_params.num_splits).
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current).  Make that
 *    first call before capturing any stream into a CUDA graph.
 *  - Sharing: every call on a device uses the same array and leaves its
 *    contents behind.  Nothing needs to start at zero (each call rewrites
 *    every value it later reads), but calls whose kernels overlap on the
 *    GPU (other streams, other host threads) race on the array: order them
 *    on one stream or serialise them. */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

pa_status pa_decode_noalloc(const pa_params *p, const void *q, const void *k_cache,
                            const void *v_cache, const int32_t *block_tables,
                            const int32_t *context_lens, float *out, uint32_t *dev_status,
                            pa_stream_t stream);

/* ----------------------------------------------------------------- prefill
 * Chunked causal prefill over packed query rows: q is [total_q][Hq][D],
 * rows cu_q_lens[s] .. cu_q_lens[s+1]-1 belong to sequence s (T_s of them),
 * cu_q_lens is [B+1] int32 on the device with cu_q_lens[0] = 0.  The chunk's
 * own K/V are already in the pages; row r attends keys 0 ..= L_s - T_s + r.
 * max_q_len is a host upper bound on every T_s (it sizes the grid);
 * total_q = cu_q_lens[B].  out is [total_q][Hq][D] f32.
 * For 16-bit Q/K/V with head_dim 64 or 128 and scale > 0 the work runs on
 * the tensor cores (tcgen05 MMA with tensor-memory accumulators); other
 * supported shapes run on the CUDA cores.  No workspace is needed
 * (pa_prefill_workspace_size returns 0; workspace may be NULL). */
size_t pa_prefill_workspace_size(const pa_params *p, int32_t total_q, int32_t max_q_len);

pa_status pa_prefill_chunk(const pa_params *p, const void *q, const int32_t *cu_q_lens,
                           int32_t total_q, int32_t max_q_len, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, float *out, void *workspace,
                           size_t workspace_bytes, uint32_t *dev_status, pa_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int32_t pa_version(void);

/* How this library was built: PA_BUILD_CHECKED when PA_CHECKED was defined
 * (kernels range-check their computed global indices; see PA_DEV_OOB). */
#define PA_BUILD_CHECKED 1
int32_t pa_build_flags(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_GQA_H */
