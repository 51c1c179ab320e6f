// Composition of partial attention results over disjoint key sets (pwwt.cn "SageAttention
// deployment pitfalls guide" §4.1: the returned log-sum-exp serves Ring Attention and similar
// schemes). One thread per (row, 8 channels): it reads the row's part LSEs, forms the weights
// exp(lse_i - max), accumulates the parts' 8 channels in fp32, and writes the normalised sum
// and the merged LSE. Memory-bound; 16-byte loads and stores where every tensor allows them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/sageattn.h"

namespace {

struct PartView {
  const void* data;
  int64_t sb, sh, sn;  // element strides of (batch, head, token)
  const float* lse;
};

struct MergeArgs {
  PartView part[SAGE_MAX_MERGE_PARTS];
  int n;
  void* out;
  int64_t ob, oh, on;
  float* lse_out;
  int heads, seqlen, d, chunks;  // chunks = ceil(d / 8)
  int64_t rows;
  int vec16;
};

template <typename T> __device__ __forceinline__ float to_float(T x);
template <> __device__ __forceinline__ float to_float<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= a.rows * a.chunks) return;
  const int64_t row = t / a.chunks;
  const int c0 = (int)(t % a.chunks) * 8;
  const int n_tok = (int)(row % a.seqlen);
  const int64_t bh = row / a.seqlen;
  const int h = (int)(bh % a.heads);
  const int64_t b = bh / a.heads;
  float w[SAGE_MAX_MERGE_PARTS];
  float m = -INFINITY;
  for (int i = 0; i < a.n; ++i) {
    w[i] = __ldg(&a.part[i].lse[row]);
    m = fmaxf(m, w[i]);
  }
  float acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = 0.f;
  float s = 0.f;
  const bool seen = m != -INFINITY;
  if (seen) {
    for (int i = 0; i < a.n; ++i) {
      const float wi = w[i] == -INFINITY ? 0.f : expf(w[i] - m);
      s += wi;
      if (wi == 0.f) continue;
      const T* src = static_cast<const T*>(a.part[i].data) + b * a.part[i].sb + h * a.part[i].sh +
                     (int64_t)n_tok * a.part[i].sn + c0;
      if (a.vec16 && c0 + 8 <= a.d) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
        const T* x = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = fmaf(wi, to_float<T>(x[c]), acc[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c0 + c < a.d) acc[c] = fmaf(wi, to_float<T>(src[c]), acc[c]);
      }
    }
  }
  const float inv = seen ? 1.0f / s : 0.f;
  T* dst = static_cast<T*>(a.out) + b * a.ob + h * a.oh + (int64_t)n_tok * a.on + c0;
  if (a.vec16 && c0 + 8 <= a.d) {
    __align__(16) T y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) y[c] = from_float<T>(acc[c] * inv);
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(y);
  } else {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c0 + c < a.d) dst[c] = from_float<T>(acc[c] * inv);
  }
  if (a.lse_out && c0 == 0) a.lse_out[row] = seen ? m + logf(s) : -INFINITY;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// element strides (batch, head, token) of a tensor in the given layout
void bhn(const sage_tensor& t, int layout, int64_t& sb, int64_t& sh, int64_t& sn) {
  sb = t.stride[0];
  if (layout == SAGE_HND) { sh = t.stride[1]; sn = t.stride[2]; }
  else { sn = t.stride[1]; sh = t.stride[2]; }
}

}  // namespace

extern "C" int sage_merge_partials(const sage_tensor* outs, const float* const* lses, int n_parts,
                                   const sage_tensor* out, float* lse_out, int batch, int heads,
                                   int seqlen, int head_dim, int dtype, int tensor_layout,
                                   void* stream) {
  if (!outs || !lses || !out || n_parts < 1 || n_parts > SAGE_MAX_MERGE_PARTS) return SAGE_ERR_INVALID_ARG;
  if (batch < 0 || heads < 0 || seqlen < 0) return SAGE_ERR_INVALID_ARG;
  if (tensor_layout != SAGE_HND && tensor_layout != SAGE_NHD) return SAGE_ERR_INVALID_ARG;
  if (dtype != SAGE_F16 && dtype != SAGE_BF16) return SAGE_ERR_DTYPE;
  if (head_dim < 1 || head_dim > 128) return SAGE_ERR_HEAD_DIM;
  MergeArgs a{};
  a.rows = (int64_t)batch * heads * seqlen;
  if (a.rows == 0) return SAGE_OK;
  a.n = n_parts;
  a.heads = heads;
  a.seqlen = seqlen;
  a.d = head_dim;
  a.chunks = (head_dim + 7) / 8;
  bool vec16 = head_dim % 8 == 0;
  for (int i = 0; i < n_parts; ++i) {
    if (!outs[i].data || !lses[i]) return SAGE_ERR_INVALID_ARG;
    if (!aligned(outs[i].data, 2) || !aligned(lses[i], 4)) return SAGE_ERR_STRIDE;
    for (int k = 0; k < 3; ++k) {
      if (outs[i].stride[k] < 0) return SAGE_ERR_STRIDE;
      vec16 = vec16 && outs[i].stride[k] % 8 == 0;
    }
    vec16 = vec16 && aligned(outs[i].data, 16);
    a.part[i].data = outs[i].data;
    a.part[i].lse = lses[i];
    bhn(outs[i], tensor_layout, a.part[i].sb, a.part[i].sh, a.part[i].sn);
  }
  if (!out->data || !aligned(out->data, 2)) return out->data ? SAGE_ERR_STRIDE : SAGE_ERR_INVALID_ARG;
  for (int k = 0; k < 3; ++k) {
    if (out->stride[k] < 0) return SAGE_ERR_STRIDE;
    vec16 = vec16 && out->stride[k] % 8 == 0;
  }
  vec16 = vec16 && aligned(out->data, 16);
  if (lse_out && !aligned(lse_out, 4)) return SAGE_ERR_STRIDE;
  a.out = out->data;
  bhn(*out, tensor_layout, a.ob, a.oh, a.on);
  a.lse_out = lse_out;
  a.vec16 = vec16 ? 1 : 0;
  const int64_t threads = a.rows * a.chunks;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return SAGE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SAGE_F16) merge_kernel<__half><<<(unsigned)blocks, 256, 0, st>>>(a);
  else merge_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}
