// pa_api.cu -- the extern "C" entry points of libpaged_gqa.so: host-side
// validation (before any device access; crucible results: malformed metadata
// is rejected before device access), the split-KV plan, workspace sizing and
// kernel dispatch.  No entry point allocates memory.
#include <math.h>
#include <string.h>

#include "pa_kernels.h"
#include "pa_prefill_f32.h"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

using pa::AttnArgs;

constexpr int kRefSms = 152;       // SM count behind the device-independent plan
constexpr int kCtasPerSm = 4;      // split-plan target: CTAs per SM
constexpr int kMinSplitPages = 1;  // smallest automatic split, in pages
constexpr int kMaxDecodeRows = 16; // query rows per sequence in pa_decode

int elt_bytes(pa_dtype d) { return d == PA_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Resolved {
    int64_t page_stride, token_stride, head_stride;
    int group;
};

pa_status check_params(const pa_params* p, Resolved* r) {
    if (!p) return PA_ERR_NULL;
    if (p->num_seqs < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1) return PA_ERR_SHAPE;
    if (p->num_seqs > 65535 || p->num_kv_heads > 65535) return PA_ERR_SHAPE;
    if (p->num_q_heads % p->num_kv_heads != 0) return PA_ERR_SHAPE;
    const int group = p->num_q_heads / p->num_kv_heads;
    if (p->q_dtype < PA_F32 || p->q_dtype > PA_BF16 || p->kv_dtype < PA_F32 ||
        p->kv_dtype > PA_BF16 || p->out_dtype < PA_F32 || p->out_dtype > PA_BF16)
        return PA_ERR_DTYPE;
    if (group > pa::kMaxGroup) return PA_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (p->page_size != 16 && p->page_size != 32) return PA_ERR_UNSUPPORTED;
    if (p->q_dtype != p->kv_dtype || p->out_dtype != PA_F32) return PA_ERR_UNSUPPORTED;
    if (p->num_pages < 1 || p->max_blocks_per_seq < 1 || p->max_context_len < 1)
        return PA_ERR_SHAPE;
    if (int64_t(p->max_context_len) > int64_t(p->max_blocks_per_seq) * p->page_size)
        return PA_ERR_SHAPE;
    if (!isfinite(p->scale)) return PA_ERR_SHAPE;
    if (p->deterministic != 0 && p->deterministic != 1) return PA_ERR_SHAPE;
    if (p->num_splits < 0) return PA_ERR_SHAPE;
    if (p->decode_phases < 0 || p->decode_phases > 3) return PA_ERR_SHAPE;
    if (p->decode_q_rows < 0 || p->decode_q_rows > kMaxDecodeRows) return PA_ERR_SHAPE;
    if (p->decode_q_rows > p->max_context_len) return PA_ERR_SHAPE;
    if (p->sliding_window < 0) return PA_ERR_SHAPE;
    if (p->decode_form < PA_FORM_AUTO || p->decode_form > PA_FORM_COUNTED) return PA_ERR_SHAPE;
    if (p->debug_timeout != 0 && p->debug_timeout != 1) return PA_ERR_SHAPE;
    const int64_t D = p->head_dim;
    r->head_stride = p->head_stride ? p->head_stride : D;
    r->token_stride = p->token_stride ? p->token_stride : p->num_kv_heads * r->head_stride;
    r->page_stride = p->page_stride ? p->page_stride : p->page_size * r->token_stride;
    if (r->head_stride < 0 || r->token_stride < 0 || r->page_stride < 0) return PA_ERR_SHAPE;
    const int eb = elt_bytes(p->kv_dtype);
    if ((r->head_stride * eb) % 16 || (r->token_stride * eb) % 16 || (r->page_stride * eb) % 16)
        return PA_ERR_ALIGN;
    r->group = group;
    return PA_OK;
}

pa_status check_io(const void* q, const void* k, const void* v, const int32_t* bt,
                   const int32_t* cl, const void* out) {
    if (!q || !k || !v || !bt || !cl || !out) return PA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PA_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(bt) & 3u) || (reinterpret_cast<uintptr_t>(cl) & 3u))
        return PA_ERR_ALIGN;
    return PA_OK;
}

int device_sms() {
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kRefSms;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = kRefSms;
        cache[dev] = n;
    }
    return cache[dev];
}

// Split plan from host fields only: splits of a whole number of pages,
// enough of them that B * Hkv * S is about kCtasPerSm CTAs per SM.
void plan(const pa_params* p, int* S, int* split_tokens) {
    const int P = p->page_size;
    const int pages = (p->max_context_len + P - 1) / P;
    int per;
    if (p->num_splits > 0) {
        per = (pages + p->num_splits - 1) / p->num_splits;
    } else {
        const int sms = p->deterministic ? kRefSms : device_sms();
        const int64_t units = int64_t(p->num_seqs) * p->num_kv_heads;
        const int64_t want = (int64_t(kCtasPerSm) * sms + units - 1) / units;
        per = int((pages + want - 1) / want);
        if (per < kMinSplitPages) per = kMinSplitPages;
    }
    if (per < 1) per = 1;
    if (per > pages) per = pages;
    *split_tokens = per * P;
    *S = (p->max_context_len + *split_tokens - 1) / *split_tokens;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// pa_decode takes the length-balanced v1 path for 16-bit K/V unless a split
// count is requested; it needs one persistent CTA per (reference) SM.
// Several query rows per sequence ride along as extra MMA columns (rows x
// q heads of a kv head <= 16).
int decode_rows(const pa_params* p) { return p->decode_q_rows > 1 ? p->decode_q_rows : 1; }

bool use_v1(const pa_params* p) {
    return p->num_splits == 0 && p->kv_dtype != PA_F32 &&
           (p->head_dim != 256 || p->num_q_heads / p->num_kv_heads <= 8);
}

// head_dim 256 runs on the split-KV kernel only (16-bit K/V, automatic
// splits, at most 8 MMA columns: rows x q heads of a kv head).
bool d256_unsupported(const pa_params* p) { return p->head_dim == 256 && !use_v1(p); }

// Rows of a split-KV unit: rows x q heads of a kv head are its MMA columns,
// at most 16 (8 at head_dim 256); more rows come in blocks of this many, each
// block its own unit of the same launch.
int row_block(const pa_params* p) {
    const int g = p->num_q_heads / p->num_kv_heads;
    const int rb = (p->head_dim == 256 ? 8 : 16) / g;
    return decode_rows(p) < rb ? decode_rows(p) : rb;
}

// The combine's grid holds one row of CTAs per (sequence, query row).
bool rows_split_ok(const pa_params* p) { return int64_t(p->num_seqs) * decode_rows(p) <= 65535; }

// Row blocks of a split-KV launch: each block of row_block rows is a unit.
int row_blocks(const pa_params* p) { return (decode_rows(p) + row_block(p) - 1) / row_block(p); }

int v1_ctas(const pa_params* p) { return p->deterministic ? kRefSms : device_sms(); }

// Split partials of every (row, q head): rows = query rows per sequence.
// They start after the counter block that pa_decode's single launch keeps at
// the head of every decode workspace, so one zeroed buffer serves both paths.
size_t partial_bytes(const pa_params* p, int S, size_t* ml_off, size_t* acc_off, int rows = 1) {
    const size_t n = size_t(p->num_seqs) * rows * p->num_q_heads * S;
    *ml_off = PA_DECODE_COUNTER_BYTES;
    *acc_off = *ml_off + align256(n * 2 * sizeof(float));
    return *acc_off + align256(n * p->head_dim * sizeof(float));
}

AttnArgs base_args(const pa_params* p, const Resolved& r, const void* q, const void* k,
                   const void* v, const int32_t* bt, const int32_t* cl, uint32_t* st) {
    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.q = q;
    a.k = k;
    a.v = v;
    a.block_tables = bt;
    a.context_lens = cl;
    a.dev_status = st;
    a.num_seqs = p->num_seqs;
    a.num_q_heads = p->num_q_heads;
    a.num_kv_heads = p->num_kv_heads;
    a.group = r.group;
    a.num_pages = p->num_pages;
    a.max_blocks_per_seq = p->max_blocks_per_seq;
    a.page_stride = r.page_stride;
    a.token_stride = r.token_stride;
    a.head_stride = r.head_stride;
    a.scale_log2 = p->scale * pa::kLog2e;
    a.total_q = p->num_seqs;
    return a;
}

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

}  // namespace

PA_EXPORT pa_params* pa_params_init(pa_params* p) {
    if (!p) return p;
    memset(p, 0, sizeof *p);
    p->out_dtype = PA_F32;
    p->deterministic = 1;
    return p;
}

PA_EXPORT const char* pa_status_string(pa_status s) {
    switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: inconsistent sizes";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: unknown dtype code";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer or stride not 16-byte aligned";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace too small";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: valid but not implemented";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA runtime call failed";
    }
    return "unknown pa_status";
}

PA_EXPORT int32_t pa_version(void) { return 200; }

PA_EXPORT int32_t pa_build_flags(void) {
#ifdef PA_CHECKED
    return PA_BUILD_CHECKED;
#else
    return 0;
#endif
}

PA_EXPORT pa_status pa_decode_plan(const pa_params* p, int32_t* num_splits, int32_t* split_tokens) {
    Resolved r;
    pa_status st = check_params(p, &r);
    if (st != PA_OK) return st;
    int S, tok;
    plan(p, &S, &tok);
    if (num_splits) *num_splits = S;
    if (split_tokens) *split_tokens = tok;
    return PA_OK;
}

PA_EXPORT size_t pa_decode_workspace_size(const pa_params* p) {
    Resolved r;
    if (check_params(p, &r) != PA_OK) return 0;
    if (d256_unsupported(p)) return 0;
    if (use_v1(p))
        return pa::decode_v1_workspace_bytes(p->num_seqs, p->num_kv_heads,
                                             row_block(p) * (p->num_q_heads / p->num_kv_heads),
                                             row_blocks(p), p->head_dim, v1_ctas(p));
    int S, tok;
    plan(p, &S, &tok);
    if (S == 1 || !rows_split_ok(p)) return 0;
    size_t ml_off, acc_off;
    return partial_bytes(p, S, &ml_off, &acc_off, decode_rows(p));
}

PA_EXPORT pa_status pa_decode_partial(const pa_params* p, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float* partial_ml,
                                      float* partial_acc, int32_t num_splits,
                                      uint32_t* dev_status, pa_stream_t stream) {
    Resolved r;
    pa_status st = check_params(p, &r);
    if (st != PA_OK) return st;
    if ((st = check_io(q, k_cache, v_cache, block_tables, context_lens, partial_ml)) != PA_OK)
        return st;
    if (!partial_acc) return PA_ERR_NULL;
    if (!aligned16(partial_acc)) return PA_ERR_ALIGN;
    if (decode_rows(p) > 1 || p->sliding_window > 0 || p->head_dim == 256) return PA_ERR_UNSUPPORTED;
    int S, tok;
    plan(p, &S, &tok);
    if (num_splits != S) return PA_ERR_SHAPE;
    AttnArgs a = base_args(p, r, q, k_cache, v_cache, block_tables, context_lens, dev_status);
    a.partial_ml = partial_ml;
    a.partial_acc = partial_acc;
    a.split_tokens = tok;
    a.num_splits = S;
    return cuda_status(pa::launch_decode_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream));
}

PA_EXPORT pa_status pa_combine(const pa_params* p, const float* partial_ml,
                               const float* partial_acc, int32_t max_splits,
                               const int32_t* splits_per_seq, float* out, pa_stream_t stream) {
    if (!p || !partial_ml || !partial_acc || !out) return PA_ERR_NULL;
    if (p->num_seqs < 1 || p->num_q_heads < 1 || max_splits < 1 || p->num_seqs > 65535 ||
        p->num_q_heads > 65535)
        return PA_ERR_SHAPE;
    if (p->head_dim == 256) return PA_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!aligned16(partial_acc) || !aligned16(out) || (reinterpret_cast<uintptr_t>(partial_ml) & 7u) ||
        (reinterpret_cast<uintptr_t>(splits_per_seq) & 3u))
        return PA_ERR_ALIGN;
    return cuda_status(pa::launch_combine_v0(partial_ml, partial_acc, out, p->num_seqs,
                                             p->num_q_heads, max_splits, p->head_dim, stream,
                                             splits_per_seq));
}

namespace {
// The split-KV kernel's call for these parameters, pointers left NULL.
pa::DecodeV1Call v1_call(const pa_params* p, const Resolved& r) {
    pa::DecodeV1Call c;
    memset(&c, 0, sizeof c);
    c.dtype = p->kv_dtype;
    c.B = p->num_seqs;
    c.Hq = p->num_q_heads;
    c.Hkv = p->num_kv_heads;
    c.D = p->head_dim;
    c.P = p->page_size;
    c.num_pages = p->num_pages;
    c.max_blocks = p->max_blocks_per_seq;
    c.n_ctas = v1_ctas(p);
    c.page_stride = r.page_stride;
    c.token_stride = r.token_stride;
    c.head_stride = r.head_stride;
    c.scale_log2 = p->scale * pa::kLog2e;
    c.phases = p->decode_phases ? p->decode_phases : 3;
    c.rows = decode_rows(p);
    c.window = p->sliding_window;
    c.row0 = 0;
    c.row_count = c.rows;
    c.row_block = row_block(p);  // blocks of rows are units of one launch
    c.single_launch = p->decode_form == PA_FORM_COUNTED;
    c.max_context_len = p->max_context_len;
    c.debug_timeout = p->debug_timeout;
    return c;
}

// pa_decode, with the new token's K/V appended first when k_new is set.
pa_status decode_impl(const pa_params* p, const void* q, const void* k_new, const void* v_new,
                      const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, float* out, void* workspace, size_t workspace_bytes,
                      uint32_t* dev_status, pa_stream_t stream) {
    Resolved r;
    pa_status st = check_params(p, &r);
    if (st != PA_OK) return st;
    if ((st = check_io(q, k_cache, v_cache, block_tables, context_lens, out)) != PA_OK) return st;
    const int rows = decode_rows(p);
    if (rows > 1 && k_new) return PA_ERR_UNSUPPORTED;  // the append takes one new token
    if (d256_unsupported(p)) return PA_ERR_UNSUPPORTED;
    if (use_v1(p)) {
        const int n = v1_ctas(p);
        const int rb = row_block(p);
        const size_t need = pa::decode_v1_workspace_bytes(p->num_seqs, p->num_kv_heads,
                                                          rb * (p->num_q_heads / p->num_kv_heads),
                                                          row_blocks(p), p->head_dim, n);
        if (!workspace) return PA_ERR_NULL;
        if (workspace_bytes < need) return PA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_ALIGN;
        pa::DecodeV1Call c = v1_call(p, r);
        c.q = q;
        c.k = k_cache;
        c.v = v_cache;
        c.block_tables = block_tables;
        c.context_lens = context_lens;
        c.out = out;
        c.workspace = workspace;
        c.dev_status = dev_status;
        c.k_new = k_new;  // fused: the partial kernel writes and attends the new rows
        c.v_new = v_new;
        return cuda_status(pa::launch_decode_v1(c, stream));
    }
    if (p->sliding_window > 0) return PA_ERR_UNSUPPORTED;  // windows: split-KV kernel only
    const int phases = p->decode_phases ? p->decode_phases : 3;
    int S, tok;
    plan(p, &S, &tok);
    if (rows > 1) {  // CUDA-core pass over row tiles x key splits, then the combine per (row, head)
        if (p->num_splits > 0) return PA_ERR_UNSUPPORTED;
        if (!rows_split_ok(p)) S = 1;
        AttnArgs a = base_args(p, r, q, k_cache, v_cache, block_tables, context_lens, dev_status);
        a.rows_per_seq = rows;
        a.max_q_len = rows;
        a.total_q = p->num_seqs * rows;
        a.num_splits = S;
        a.split_tokens = tok;
        if (S == 1) {
            a.out = out;
            if (!(phases & 1)) return PA_OK;
            return cuda_status(pa::launch_prefill_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream));
        }
        size_t ml_off, acc_off;
        const size_t need = partial_bytes(p, S, &ml_off, &acc_off, rows);
        if (!workspace) return PA_ERR_NULL;
        if (workspace_bytes < need) return PA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_ALIGN;
        a.partial_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off);
        a.partial_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_off);
        if (phases & 1) {
            cudaError_t e = pa::launch_prefill_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream);
            if (e != cudaSuccess) return PA_ERR_CUDA;
        }
        if (!(phases & 2)) return PA_OK;
        return cuda_status(pa::launch_combine_v0(a.partial_ml, a.partial_acc, out, p->num_seqs * rows,
                                                 p->num_q_heads, S, p->head_dim, stream));
    }
    if (k_new && (!p->decode_phases || (p->decode_phases & 1))) {
        cudaError_t e = pa::launch_append_kv(k_new, v_new, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                             block_tables, context_lens, p->num_seqs, p->num_kv_heads,
                                             p->head_dim, p->page_size, p->kv_dtype == PA_F32 ? 4 : 2,
                                             p->num_pages, p->max_blocks_per_seq, r.page_stride,
                                             r.token_stride, r.head_stride, stream);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    AttnArgs a = base_args(p, r, q, k_cache, v_cache, block_tables, context_lens, dev_status);
    a.split_tokens = tok;
    a.num_splits = S;
    if (S == 1) {
        a.out = out;
        if (!(phases & 1)) return PA_OK;
        return cuda_status(pa::launch_decode_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream));
    }
    size_t ml_off, acc_off;
    const size_t need = partial_bytes(p, S, &ml_off, &acc_off);
    if (!workspace) return PA_ERR_NULL;
    if (workspace_bytes < need) return PA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_ALIGN;
    a.partial_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off);
    a.partial_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_off);
    if (phases & 1) {
        cudaError_t e = pa::launch_decode_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    if (!(phases & 2)) return PA_OK;
    return cuda_status(pa::launch_combine_v0(a.partial_ml, a.partial_acc, out, p->num_seqs,
                                             p->num_q_heads, S, p->head_dim, stream));
}
}  // namespace

PA_EXPORT int32_t pa_decode_kernels(const pa_params* p, int32_t with_append) {
    Resolved r;
    if (check_params(p, &r) != PA_OK || d256_unsupported(p)) return -1;
    const int phases = p->decode_phases ? p->decode_phases : 3;
    if (use_v1(p)) {
        pa::DecodeV1Call c = v1_call(p, r);
        if (with_append) c.k_new = c.v_new = &c;  // only marks the append (the plan has no small-call form for it)
        return pa::decode_v1_kernels(c);
    }
    if (p->sliding_window > 0 || (with_append && decode_rows(p) > 1)) return -1;
    int S, tok;
    plan(p, &S, &tok);
    if (decode_rows(p) > 1 && !rows_split_ok(p)) S = 1;
    const int scatter = with_append && (phases & 1) ? 1 : 0;  // the append's scatter kernel
    if (S == 1) return (phases & 1) ? 1 + scatter : 0;
    return ((phases & 1) ? 1 + scatter : 0) + ((phases & 2) ? 1 : 0);
}

PA_EXPORT pa_status pa_decode(const pa_params* p, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              const int32_t* context_lens, float* out, void* workspace,
                              size_t workspace_bytes, uint32_t* dev_status, pa_stream_t stream) {
    return decode_impl(p, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens, out,
                       workspace, workspace_bytes, dev_status, stream);
}

PA_EXPORT pa_status pa_decode_append(const pa_params* p, const void* q, const void* k_new,
                                     const void* v_new, void* k_cache, void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     float* out, void* workspace, size_t workspace_bytes,
                                     uint32_t* dev_status, pa_stream_t stream) {
    if (!k_new || !v_new) return PA_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new)) return PA_ERR_ALIGN;
    return decode_impl(p, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out,
                       workspace, workspace_bytes, dev_status, stream);
}

PA_EXPORT size_t pa_prefill_workspace_size(const pa_params* p, int32_t total_q, int32_t max_q_len) {
    (void)p;
    (void)total_q;
    (void)max_q_len;
    return 0;
}

PA_EXPORT pa_status pa_prefill_chunk(const pa_params* p, const void* q, const int32_t* cu_q_lens,
                                     int32_t total_q, int32_t max_q_len, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, float* out, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_status,
                                     pa_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    Resolved r;
    pa_status st = check_params(p, &r);
    if (st != PA_OK) return st;
    if ((st = check_io(q, k_cache, v_cache, block_tables, context_lens, out)) != PA_OK) return st;
    if (!cu_q_lens) return PA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u) return PA_ERR_ALIGN;
    if (total_q < 1 || max_q_len < 1 || max_q_len > p->max_context_len) return PA_ERR_SHAPE;
    if (p->sliding_window > 0 || p->head_dim == 256) return PA_ERR_UNSUPPORTED;  // decode only
    AttnArgs a = base_args(p, r, q, k_cache, v_cache, block_tables, context_lens, dev_status);
    a.cu_q_lens = cu_q_lens;
    a.out = out;
    a.max_q_len = max_q_len;
    a.total_q = total_q;
    a.num_splits = 1;
    a.debug_timeout = p->debug_timeout;
    if (pa::prefill_tc_supported(p->kv_dtype, p->head_dim, p->page_size, r.group, p->scale))
        return cuda_status(pa::launch_prefill_tc(a, p->kv_dtype, p->head_dim, p->page_size, stream));
    if (p->kv_dtype == PA_F32 && pa::prefill_f32_supported(p->head_dim, p->page_size, r.group))
        return cuda_status(pa::launch_prefill_f32(a, p->head_dim, p->page_size, stream));
    return cuda_status(pa::launch_prefill_v0(a, p->kv_dtype, p->head_dim, p->page_size, stream));
}
