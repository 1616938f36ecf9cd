// pa_kernels.h -- launchers of the CUDA kernels (internal to the library).
#pragma once

#include "pa_common.cuh"

namespace pa {

// v0 tile kernel: decode split partials (a.out == nullptr) or the final
// output (a.out set, single split); grid (S, Hkv, B).
cudaError_t launch_decode_v0(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st);
// v0 tile kernel over packed prefill rows; grid (ceil(max_q_len/4), Hkv, B).
cudaError_t launch_prefill_v0(const AttnArgs& a, pa_dtype dt, int D, int P, cudaStream_t st);
// Split combine, grid (Hq, B), D threads.
cudaError_t launch_combine_v0(const float* ml, const float* acc, float* out, int B, int Hq,
                              int S, int D, cudaStream_t st);

}  // namespace pa
