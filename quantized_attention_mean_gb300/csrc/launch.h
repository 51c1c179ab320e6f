// Host-side launchers of the kernels (defined next to each kernel).
#pragma once
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include "problem.cuh"

namespace sage {
// Programmatic dependent launch: the kernel may start while the previous kernel in the
// stream is finishing; it must execute pdl_wait() before it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device,
// calling the runtime only when the limit recorded for that device is lower (the same kernel is
// launched on every call). `limits` is one per kernel: the largest value set on each device.
template <typename K>
cudaError_t raise_smem_limit(K* kernel, int bytes, std::atomic<int> (&limits)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  }
  if (limits[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    int cur = limits[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !limits[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

// Records a failed CUDA call for sage_last_cuda_error (calling thread) and returns
// SAGE_ERR_CUDA.
int note_cuda_failure(cudaError_t e, const char* where);

cudaError_t launch_varlen_setup(const Problem& p, cudaStream_t st);
cudaError_t launch_kv_stats(const Problem& p, int max_len_k, cudaStream_t st);
cudaError_t launch_short_status_clear(int* err, int words, cudaStream_t st);
cudaError_t launch_finalize(const Problem& p, int n_stats, cudaStream_t st);
cudaError_t launch_quant(const Problem& p, int max_len_q, int max_len_k, cudaStream_t st);
cudaError_t launch_export_codes(const __half* codes, int64_t rows_pp, int dp, int d, int planes,
                                int n, int8_t* out, cudaStream_t st);
cudaError_t launch_export_vt(const uint8_t* vt, int64_t pitch, int dp, int d, int planes, int n,
                             uint8_t* out, cudaStream_t st);
cudaError_t launch_e4m3(const float* x, uint8_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_e2m1(const float* x, uint8_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_export_fp16(const __half* codes, int64_t rows_pp, int dp, int d, int planes,
                               int n, uint16_t* out, cudaStream_t st);
cudaError_t launch_export_vt16(const __half* vt, int64_t pitch, int dp, int d, int planes, int n,
                               uint16_t* out, cudaStream_t st);
// Short-sequence kernel: one launch for the whole forward of a dense problem with at most
// kShortMaxKeys keys and kShortMaxQueries queries (statistics, quantisation and attention per
// CTA of 128 query rows; short.cu). Selected with sage_debug_select_path(2).
constexpr int kShortMaxKeys = 256, kShortMaxQueries = 1024;
cudaError_t launch_short_attention(const Problem& p, cudaStream_t st);

cudaError_t launch_attention(const Problem& p, const CUtensorMap* maps, int grid_pairs,
                             cudaStream_t stream);
}  // namespace sage
