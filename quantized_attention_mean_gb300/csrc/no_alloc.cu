// sage_attn_no_alloc: the dense forward for callers that cannot allocate device memory.
//
// Some callers own no allocator at the point where they run attention: a plugin executing
// inside a host engine that hands it only its input and output buffers and forbids device
// allocation while the engine is running, or a latency-critical path where neither the
// time of a cudaMalloc nor the chance of it failing is acceptable. For them this entry
// point takes the scratch memory sage_attn needs from a fixed-size array that is part of
// the library image (every GPU that loads the library holds it until the process exits).
// The caller still passes its inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sageattn.h"
#include "launch.h"

namespace {

// Scratch memory of sage_attn_no_alloc, shared by every call on a device.
static __device__ __align__(256) unsigned char g_scratch[SAGE_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device

// Device address of the scratch array on the current device. In host code g_scratch names
// a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached. On failure the runtime's error is taken off the thread (so that no
// later launch check reports it as its own) and recorded for sage_last_cuda_error;
// returns nullptr.
void* scratch_address() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    sage::note_cuda_failure(e != cudaSuccess ? e : cudaErrorInvalidDevice, "no-alloc scratch: device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      sage::note_cuda_failure(e, "no-alloc scratch: cudaGetSymbolAddress");
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int sage_attn_no_alloc(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                                  const sage_tensor* out, float* lse, int batch, int heads_q,
                                  int heads_kv, int seqlen_q, int seqlen_k, int head_dim,
                                  int dtype, int tensor_layout, int is_causal, float sm_scale,
                                  int return_lse, int qk_quant_gran, int pv_accum_dtype,
                                  int smooth_k, int smooth_v, void* stream) {
  // Argument checks first, with sage_attn's own rules and codes: without a workspace it
  // validates everything else and launches nothing (an empty problem returns SAGE_OK, a
  // valid one SAGE_ERR_WORKSPACE).
  const int st = sage_attn(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k,
                           head_dim, dtype, tensor_layout, is_causal, sm_scale, return_lse,
                           qk_quant_gran, pv_accum_dtype, smooth_k, smooth_v, nullptr, 0, stream);
  if (st != SAGE_ERR_WORKSPACE) return st;
  const size_t need = sage_attn_workspace_size(batch, heads_q, heads_kv, seqlen_q, seqlen_k,
                                               head_dim, qk_quant_gran);
  if (need > SAGE_NO_ALLOC_SCRATCH_BYTES) return SAGE_ERR_WORKSPACE;
  if (!sage_device_supported()) return SAGE_ERR_DEVICE;
  void* scratch = scratch_address();
  if (scratch == nullptr) return SAGE_ERR_CUDA;
  // The statistics and status regions are cleared by the call itself; nothing left in the
  // scratch by an earlier call is read.
  return sage_attn(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim,
                   dtype, tensor_layout, is_causal, sm_scale, return_lse, qk_quant_gran,
                   pv_accum_dtype, smooth_k, smooth_v, scratch, SAGE_NO_ALLOC_SCRATCH_BYTES,
                   stream);
}
