// pa_prefill_f32.h -- launcher of the register-tiled fp32 chunked prefill.
#pragma once

#include "pa_common.cuh"

namespace pa {

// Chunked causal prefill with fp32 Q/K/V (out = final rows, no split
// partials): head_dim 64 or 128, page size 16 or 32, Hq / Hkv <= 16.
bool prefill_f32_supported(int D, int P, int G);
cudaError_t launch_prefill_f32(const AttnArgs& a, int D, int P, cudaStream_t st);

}  // namespace pa
