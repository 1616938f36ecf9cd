// pa_noalloc.cu -- pa_decode for callers that cannot allocate device memory.
//
// pa_decode needs a caller-provided workspace for its split partials.  Some
// callers have no way to obtain one at call time: an inference-engine plugin
// whose host owns every device buffer, a serving loop that forbids
// allocation after start-up, or a process whose caching allocator already
// holds all free memory.  pa_decode_noalloc keeps the partials in a fixed
// array that lives in this library's device image instead, so the caller
// passes only inputs and outputs.  It runs the same kernels as pa_decode,
// through pa_decode_partial and pa_combine.
#include <mutex>

#include "pa_common.cuh"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

// The scratch itself: allocated when the library's device code is loaded on
// a GPU and held until the process exits.  In host code `g_noalloc_scratch`
// names a host-side stand-in, not the device address; the device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of the array, per device

// Device address of the scratch on the current device, looked up once per
// device (with that device current).
pa_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

PA_EXPORT pa_status pa_decode_noalloc(const pa_params* p, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float* out,
                                      uint32_t* dev_status, pa_stream_t stream) {
    int32_t S = 0, split_tokens = 0;
    pa_status st = pa_decode_plan(p, &S, &split_tokens);
    if (st != PA_OK) return st;
    // Everything the host can check is checked before the partial step is
    // enqueued: the output pointer (the partial step does not see it) and the
    // options the fixed split plan does not take.
    if (!out) return PA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(out) & 15u) return PA_ERR_ALIGN;
    if (p->decode_q_rows > 1 || p->sliding_window > 0 || p->head_dim == 256) return PA_ERR_UNSUPPORTED;
    // partial layout: m/l pairs, then the 256-byte aligned accumulators
    const size_t n = size_t(p->num_seqs) * p->num_q_heads * S;
    const size_t acc_off = round256(n * 2 * sizeof(float));
    const size_t need = acc_off + n * size_t(p->head_dim) * sizeof(float);
    if (need > size_t(PA_NOALLOC_SCRATCH_BYTES)) return PA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != PA_OK) return st;
    float* ml = static_cast<float*>(scratch);
    float* acc = reinterpret_cast<float*>(static_cast<char*>(scratch) + acc_off);
    // Every (m, l) pair is rewritten by the partial step and an accumulator is
    // read only when its m is finite, so stale contents never reach `out`.
    st = pa_decode_partial(p, q, k_cache, v_cache, block_tables, context_lens, ml, acc, S,
                           dev_status, stream);
    if (st != PA_OK) return st;
    return pa_combine(p, ml, acc, S, nullptr, out, stream);
}
