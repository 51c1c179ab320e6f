// Host-side launchers of the kernels (defined next to each kernel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "problem.cuh"

namespace sage {
cudaError_t launch_varlen_setup(const Problem& p, cudaStream_t st);
cudaError_t launch_kv_stats(const Problem& p, int max_len_k, cudaStream_t st);
cudaError_t launch_finalize(const Problem& p, int n_stats, cudaStream_t st);
cudaError_t launch_quant(const Problem& p, int max_len_q, int max_len_k, cudaStream_t st);
cudaError_t launch_export_codes(const __half* codes, int64_t rows_pp, int dp, int d, int planes,
                                int n, int8_t* out, cudaStream_t st);
cudaError_t launch_export_vt(const uint8_t* vt, int64_t pitch, int dp, int d, int planes, int n,
                             uint8_t* out, cudaStream_t st);
cudaError_t launch_e4m3(const float* x, uint8_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_attention(const Problem& p, const CUtensorMap* maps, int grid_pairs,
                             cudaStream_t stream);
}  // namespace sage
