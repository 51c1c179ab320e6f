// Stages 1-2 of the method (pwwt.cn "SageAttention deployment pitfalls guide" §1, §4.2):
// smoothing statistics for K and V, INT8 quantisation of Q and K with per-token-group
// scales, and per-channel FP8 E4M3 quantisation of V.
//
// Both kernels are HBM-bound streaming passes: each block walks a tile of tokens with
// 16-byte vector loads (8 channels per thread, head_dim / 8 threads per token row), reduces
// with warp shuffles and shared memory, and writes coalesced outputs.
//
// Bit-exactness: the mean is an exact fixed-point sum (order-free, so atomics are fine);
// scales and codes use explicitly rounded IEEE operations: scalar __fdiv_rn, __fmul_rn,
// __fadd_rn / __fsub_rn, and packed f32x2 operations only where no multiply is followed by an
// add (the compiler may fuse a packed multiply and add into one packed fma), so no
// contraction or reassociation can change a code.
#include "launch.h"
#include "problem.cuh"
#include "sm103_ptx.cuh"

namespace sage {

// Two 16-bit floats of one input word as fp32 (low half first), exactly.
template <typename T> __device__ __forceinline__ void unpack2(uint32_t w, float& a, float& b);
template <> __device__ __forceinline__ void unpack2<__nv_bfloat16>(uint32_t w, float& a, float& b) {
  a = __uint_as_float(w << 16);
  b = __uint_as_float(w & 0xFFFF0000u);
}
template <> __device__ __forceinline__ void unpack2<__half>(uint32_t w, float& a, float& b) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
  a = f.x;
  b = f.y;
}
// Lane-wise min / max / larger magnitude of two raw fp16 or bf16 pairs (exact; a NaN lane
// yields the other operand, as fminf / fmaxf do; the magnitude form's sign bits are not used).
template <typename T> __device__ __forceinline__ uint32_t hmin2_raw(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (std::is_same<T, __half>::value) asm("min.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <typename T> __device__ __forceinline__ uint32_t hmax2_raw(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (std::is_same<T, __half>::value) asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <typename T> __device__ __forceinline__ uint32_t habsmax2_raw(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (std::is_same<T, __half>::value)
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_s16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------------------------------
// Varlen set-up: validate cu_seqlens and lay sequences out in 128-row aligned segments.
// One block. Writes seqinfo (tok0, len, row0 for q and k, LPT order); invalid input
// records kDevSeqlens and zeroes every length so later kernels do nothing.
__global__ void __launch_bounds__(1024) varlen_setup_kernel(Problem p) {
  const int B = p.batch;
  int* si = p.seqinfo;
  __shared__ int bad;
  if (threadIdx.x == 0) {
    bad = 0;
    if (p.cu_q[0] != 0 || p.cu_k[0] != 0 || p.cu_q[B] != p.total_q || p.cu_k[B] != p.total_k)
      bad = 1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int lq = p.cu_q[b + 1] - p.cu_q[b], lk = p.cu_k[b + 1] - p.cu_k[b];
    if (lq < 0 || lk < 0 || lq > p.nq || lk > p.nk || (lq > 0 && lk == 0)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int rq = 0, rk = 0;
    for (int b = 0; b < B; ++b) {
      const int lq = bad ? 0 : p.cu_q[b + 1] - p.cu_q[b];
      const int lk = bad ? 0 : p.cu_k[b + 1] - p.cu_k[b];
      si[kSiTok0Q * B + b] = bad ? 0 : p.cu_q[b];
      si[kSiLenQ * B + b] = lq;
      si[kSiRow0Q * B + b] = rq;
      si[kSiTok0K * B + b] = bad ? 0 : p.cu_k[b];
      si[kSiLenK * B + b] = lk;
      si[kSiRow0K * B + b] = rk;
      rq += (lq + kTileRows - 1) / kTileRows * kTileRows;
      rk += (lk + kTileKeys - 1) / kTileKeys * kTileKeys;
    }
    if (bad) record_error(p.err, kDevSeqlens);
  }
  __syncthreads();
  // Longest-processing-time order: sequences by decreasing len_q * len_k (stable).
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const long long w = (long long)si[kSiLenQ * B + b] * si[kSiLenK * B + b];
    int rank = 0;
    if (B <= 4096) {
      for (int o = 0; o < B; ++o) {
        const long long wo = (long long)si[kSiLenQ * B + o] * si[kSiLenK * B + o];
        rank += (wo > w) || (wo == w && o < b);
      }
    } else {
      rank = b;
    }
    si[kSiOrder * B + rank] = b;
  }
}

// ------------------------------------------------------------------------------------------
// K/V statistics of one block of tokens (KIND 0: K, the fixed-point sum, run only with
// smooth_k; KIND 1: V, the fixed-point sum with smooth_v, and the min / max). Per (sequence,
// kv head, channel). Grid: (token chunks, Hkv, batch). 256 threads: thread = (row group rg,
// channel vector vec); TPR = padded head_dim / 8 threads per row. A block walks nb <= 4
// batches of 4 rows per thread (rows rg + RG * i), the next batch's loads in flight while the
// current one is summed.
//
// Fixed-point sum, fast form (every |x| < 2^14 and, for bf16, no nonzero |x| < 2^-17, so that
// x * 2^24 is an integer): hacc runs as 1.5 * 2^23 + sum(h), where h = round(16 x) is taken
// against hacc itself (t = fl(hacc + 16 x), h = t - hacc, both exact in the binade
// [2^23, 2^24) because a thread's at most 16 rows keep |sum h| <= 2^22), and racc sums the
// exact remainders r = 16 x - h (|r| <= 1/2 on the 2^-20 lattice, |sum r| <= 8). Warps that
// see any other value redo their rows with exact int64 conversions.
template <typename T, int TPR, int KIND>
__device__ __forceinline__ void kv_stats_block(const Problem& p, int chunk, int hk, int b, int nb) {
  constexpr int RG = 256 / TPR;
  constexpr bool kBf16 = !std::is_same<T, __half>::value;
  const Seq s = get_seq(p, b);
  const int t0 = chunk * RG * 4 * nb;
  if (t0 >= s.len_k) return;
  const int t1 = min(t0 + RG * 4 * nb, s.len_k);
  const int vec = threadIdx.x % TPR, rg = threadIdx.x / TPR;
  const int c0 = vec * 8;
  const bool active = c0 < p.d;
  const bool want_sum = KIND == 0 || p.smooth_v;
  const T* base = KIND == 0
      ? static_cast<const T*>(p.k) + (int64_t)b * p.k_sb + (int64_t)hk * p.k_sh
      : static_cast<const T*>(p.v) + (int64_t)b * p.v_sb + (int64_t)hk * p.v_sh;
  const int64_t sn = KIND == 0 ? p.k_sn : p.v_sn;
  // packed 16-bit accumulators over raw input words (two channels each): V's min / max, K's
  // max |x|, and (bf16) the smallest nonzero magnitude, kept as the signed 16-bit value
  // (|x| bits | 0x8000) - 1 so that zero maps to the largest one
  uint32_t mn[4], mx[4], ax[4], nz[4];
  float hacc[8], racc[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mn[j] = kBf16 ? 0x7F807F80u : 0x7C007C00u;  // +inf pairs
    mx[j] = kBf16 ? 0xFF80FF80u : 0xFC00FC00u;  // -inf pairs
    ax[j] = 0u;
    nz[j] = 0x7FFF7FFFu;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    hacc[i] = kRoundMagic;
    racc[i] = 0.f;
  }

  auto load_batch = [&](int k, uint4 (&dst)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = t0 + rg + RG * (4 * k + i);
      dst[i] = (active && t < t1) ? load8_raw<T>(base + (int64_t)(s.tok0_k + t) * sn, c0, p.d, p.vec16)
                                  : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 cur[4], nxt[4] = {};
  load_batch(0, cur);
  for (int k = 0; k < nb; ++k) {
    if (k + 1 < nb) load_batch(k + 1, nxt);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool live = t0 + rg + RG * (4 * k + i) < t1;
      const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (KIND == 1 && live) {
          mn[j] = hmin2_raw<T>(mn[j], w[j]);
          mx[j] = hmax2_raw<T>(mx[j], w[j]);
        }
        if (want_sum) {
          if (KIND == 0) ax[j] = habsmax2_raw<T>(ax[j], w[j]);
          if (kBf16) nz[j] = min_s16x2(nz[j], (w[j] | 0x80008000u) - 0x00010001u);
          float x0, x1, t0f, t1f, n0, n1, r0, r1;
          unpack2<T>(w[j], x0, x1);
          fma2(t0f, t1f, x0, x1, 16.0f, 16.0f, hacc[2 * j], hacc[2 * j + 1]);  // hacc + round(16 x)
          fma2(n0, n1, t0f, t1f, -1.0f, -1.0f, hacc[2 * j], hacc[2 * j + 1]);  // -round(16 x)
          fma2(r0, r1, x0, x1, 16.0f, 16.0f, n0, n1);                          // exact remainder
          add2(racc[2 * j], racc[2 * j + 1], racc[2 * j], racc[2 * j + 1], r0, r1);
          hacc[2 * j] = t0f;
          hacc[2 * j + 1] = t1f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
  }

  // largest magnitude (range check and fast-form bound) and the bf16 small-value test
  float amax = 0.f;
  bool fast = true;
  const bool seen = active && t0 + rg < t1;  // V: this thread's min / max hold a row
  if (want_sum) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a0, a1, b0, b1;
      if (KIND == 0) {
        unpack2<T>(ax[j], a0, a1);
        amax = fmaxf(amax, fmaxf(fabsf(a0), fabsf(a1)));
      } else if (seen) {
        unpack2<T>(mn[j], a0, a1);
        unpack2<T>(mx[j], b0, b1);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))));
      }
      // a nonzero bf16 magnitude below 2^-17 (bits 1 .. 0x36FF) leaves a value below
      // -32768 + 0x36FF in its half of nz
      if (kBf16)
        fast &= static_cast<int16_t>(nz[j] & 0xFFFFu) >= -32768 + 0x36FF &&
                static_cast<int16_t>(nz[j] >> 16) >= -32768 + 0x36FF;
    }
    fast &= amax < 16384.0f;
    const float lim = p.varlen ? __shfl_sync(0xffffffffu,
                                             (threadIdx.x & 31) == 0
                                                 ? __double2float_ru(__ddiv_rn(274877906944.0, (double)s.len_k))
                                                 : 0.f,
                                             0)
                               : p.range_limit;
    if (amax >= lim) record_error(p.err, kDevRange);
  }
  // sum(x * 2^24) = 2^20 sum(h) + 2^20 sum(r): |sum h| <= 2^22 sits in hacc's low mantissa
  // bits, and 2^20 sum(r) (an integer, at most 2^23) converts exactly
  long long sum[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    sum[i] = (static_cast<long long>(static_cast<int>(__float_as_uint(hacc[i]) - kRoundMagicBits)) << 20) +
             __float2int_rn(__fmul_rn(racc[i], 1048576.0f));
  if (want_sum && !__all_sync(0xffffffffu, fast)) {
    // exact int64 conversion of every row of this warp's threads instead
#pragma unroll
    for (int i = 0; i < 8; ++i) sum[i] = 0;
    if (active) {
      for (int r = 0; r < 4 * nb; ++r) {
        const int t = t0 + rg + RG * r;
        if (t >= t1) continue;
        float x[8];
        unpack8<T>(load8_raw<T>(base + (int64_t)(s.tok0_k + t) * sn, c0, p.d, p.vec16), x);
#pragma unroll
        for (int i = 0; i < 8; ++i) sum[i] += __float2ll_rz(x[i] * 16777216.0f);
      }
    }
  }
  float fmn[8], fmx[8];
  if (KIND == 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      unpack2<T>(mn[j], fmn[2 * j], fmn[2 * j + 1]);
      unpack2<T>(mx[j], fmx[2 * j], fmx[2 * j + 1]);
    }
  }
  // reduce the row groups that share a warp, then the 8 warps through shared memory
#pragma unroll
  for (int off = TPR; off < 32; off <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (want_sum) sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], off);
      if (KIND == 1) {
        fmn[i] = fminf(fmn[i], __shfl_xor_sync(0xffffffffu, fmn[i], off));
        fmx[i] = fmaxf(fmx[i], __shfl_xor_sync(0xffffffffu, fmx[i], off));
      }
    }
  }
  __shared__ long long red_s[8][128];
  __shared__ float red_f[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t sidx = ((int64_t)b * p.hkv + hk) * p.d;
  if (want_sum) {
    if (lane < TPR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) red_s[warp][c0 + i] = sum[i];
    }
    __syncthreads();
    if (threadIdx.x < p.d) {
      long long acc = 0;
      for (int w = 0; w < 8; ++w) acc += red_s[w][threadIdx.x];
      atomicAdd(reinterpret_cast<unsigned long long*>(KIND == 0 ? &p.ksum[sidx + threadIdx.x]
                                                                 : &p.vsum[sidx + threadIdx.x]),
                static_cast<unsigned long long>(acc));
    }
  }
  if (KIND == 1) {
    if (lane < TPR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) red_f[warp][c0 + i] = fmn[i];
    }
    __syncthreads();
    if (threadIdx.x < p.d) {
      float m = red_f[0][threadIdx.x];
      for (int w = 1; w < 8; ++w) m = fminf(m, red_f[w][threadIdx.x]);
      atomicMax(&p.vmin[sidx + threadIdx.x], ~ordered_code(m));
    }
    __syncthreads();
    if (lane < TPR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) red_f[warp][c0 + i] = fmx[i];
    }
    __syncthreads();
    if (threadIdx.x < p.d) {
      float m = red_f[0][threadIdx.x];
      for (int w = 1; w < 8; ++w) m = fmaxf(m, red_f[w][threadIdx.x]);
      atomicMax(&p.vmax[sidx + threadIdx.x], ordered_code(m));
    }
  }
}

// Both tensors' statistics in one launch. Grid: (token chunks, Hkv, batch x tensors): blockIdx.z
// = b + batch * t, t = 0 for K (present only with smooth_k) and the last t for V; each chunk
// is nb batches of 4 * RG tokens.
template <typename T, int TPR>
__global__ void __launch_bounds__(256, 3) kv_stats_kernel(Problem p, int nb) {
  pdl_trigger();
  const int b = blockIdx.z % p.batch;
  const bool is_k = p.smooth_k && (int)blockIdx.z < p.batch;
  if (is_k) kv_stats_block<T, TPR, 0>(p, blockIdx.x, blockIdx.y, b, nb);
  else kv_stats_block<T, TPR, 1>(p, blockIdx.x, blockIdx.y, b, nb);
}

// ------------------------------------------------------------------------------------------
// Per (sequence, kv head, channel): the smoothing means from the fixed-point sums, and V's
// per-channel scale s_v = fl32(absmax/448) and reciprocal fl32(448/absmax), where
// absmax = max(|fl32(vmax - vmean)|, |fl32(vmin - vmean)|) (x -> fl32(x - m) is monotone, so
// this equals the max over tokens of |fl32(v - vmean)|). Computed once here so the
// quantisation pass needs no double-precision arithmetic.
__global__ void kv_finalize_kernel(Problem p, int n_stats) {
  pdl_trigger();
  pdl_wait();  // the statistics kernel's sums
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_stats) return;
  const int b = i / (p.hkv * p.d);
  const Seq s = get_seq(p, b);
  if (s.len_k <= 0) return;
  const float km = p.smooth_k ? fixed_point_mean(p.ksum[i], s.len_k) : 0.f;
  const float vm = p.smooth_v ? fixed_point_mean(p.vsum[i], s.len_k) : 0.f;
  const float mx = __fsub_rn(ordered_decode(p.vmax[i]), vm);
  const float mn = __fsub_rn(ordered_decode(~p.vmin[i]), vm);
  const float amax = fmaxf(fabsf(mx), fabsf(mn));
  p.kmean[i] = km;
  p.vmean[i] = vm;
  // the FP16 P·V variant keeps V' unscaled; the FP8 and FP4 ones map absmax onto 448
  const bool unscaled = p.pv16 && !p.fp4;
  p.vscale[i] = unscaled ? 1.0f : (amax > 0.f ? __fdiv_rn(amax, 448.0f) : 0.f);
  p.vrcp[i] = unscaled ? 1.0f : (amax > 0.f ? __fdiv_rn(448.0f, amax) : 0.f);
}

// ------------------------------------------------------------------------------------------
// Quantisation, one instantiation per tensor (kind 0 = Q, 1 = K, 2 = V, 3 = V in fp16;
// FP4 variant: 4 = Q, 5 = K, 6 = V). Grid: (128-token
// tiles, heads, batch). NT threads; thread (rg, vec) holds rows rg + RG*i (i < 128 / RG,
// RG = NT / TPR), channels [8*vec, 8*vec + 8). NT is 512 for dense problems at padded
// head_dim 128 (4 rows per thread: less unrolled code per warp than 8 rows at 256 threads,
// measured 7-17% faster) and 256 otherwise (at head_dim 64, 2 rows per thread measured slower;
// varlen grids hold many empty tiles, which cost more at 512).
//   Q: codes = INT8 per group of gq rows (stored as integer-valued fp16 for the tensor
//      cores), scales sq, and (return_lse with smooth_k) the LSE term q . kmean.
//   K: K' = K - kmean, INT8 per group of gk rows.
//   V: V' = V - vmean, E4M3 with the per-channel scale absmax/448, written transposed
//      [channel][token] so that P.V reads V^T tiles K-major.
//   V (kind 3, FP16 P·V variant): V' = V - vmean rounded to fp16 (RNE), transposed likewise.
//   FP4 variant: Q and K' (kinds 4, 5) are mapped onto [-448, 448] by their token group's
//      scale g = absmax/448 (u = fl32(x · fl32(448/absmax))) and microscaled in blocks of 16
//      channels of a row; V' (kind 6) is mapped by its channel's scale (as for FP8) and
//      microscaled in blocks of 16 tokens of a channel, transposed like kind 3. Each element
//      is stored as its fp16 carrier (E2M1 code x E4M3 block scale).
// Rows past the sequence end up to the stored tile end are written as zeros.
template <typename T, int kind, int TPR, int NT>
__device__ __forceinline__ void quant_block(const Problem& p, int tile, int h, int b) {
  constexpr int RG = NT / TPR;       // row groups
  constexpr int RPT = kTileRows / RG;  // rows per thread
  const Seq s = get_seq(p, b);
  const int len = (kind == 0 || kind == 4) ? s.len_q : s.len_k;
  // rows stored for this sequence: dense planes hold exactly len rows; varlen segments are
  // padded to a multiple of 128
  const int stored = p.varlen ? (len + kTileRows - 1) / kTileRows * kTileRows : len;
  const int r0 = tile * kTileRows;
  if (r0 >= stored) return;
  const int vec = threadIdx.x % TPR, rg = threadIdx.x / TPR;
  const int c0 = vec * 8;
  const int d = p.d, dp = p.dp;
  const int hk = (kind == 0 || kind == 4) ? h / (p.hq / p.hkv) : h;  // kv head of this q head
  const int64_t sidx = ((int64_t)b * p.hkv + hk) * d;

  __shared__ float rowmax[kTileRows];
  __shared__ float grcp[kTileRows];

  // per-channel values from the finalize pass: smoothing means, V scale reciprocals, and for
  // Q heads the K mean used by the LSE term
  constexpr bool kIsQ = kind == 0 || kind == 4, kIsK = kind == 1 || kind == 5;
  constexpr bool kIsV = !kIsQ && !kIsK;
  float mean[8], rcpv[8], kmean_q[8];
  const bool want_qkc = kIsQ && p.return_lse && p.smooth_k;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool ch = c0 + i < d;
    mean[i] = (ch && kIsK) ? p.kmean[sidx + c0 + i] : ((ch && kIsV) ? p.vmean[sidx + c0 + i] : 0.f);
    rcpv[i] = (ch && (kind == 2 || kind == 6)) ? p.vrcp[sidx + c0 + i] : 0.f;
    kmean_q[i] = (ch && want_qkc) ? p.kmean[sidx + c0 + i] : 0.f;
  }

  // load the tile as raw 16-byte words (values past the sequence end and channels past d are
  // 0); every row of the thread is requested before any is used
  const T* base;
  int64_t sn;
  if (kIsQ) {
    base = static_cast<const T*>(p.q) + (int64_t)b * p.q_sb + (int64_t)h * p.q_sh; sn = p.q_sn;
  } else if (kIsK) {
    base = static_cast<const T*>(p.k) + (int64_t)b * p.k_sb + (int64_t)h * p.k_sh; sn = p.k_sn;
  } else {
    base = static_cast<const T*>(p.v) + (int64_t)b * p.v_sb + (int64_t)h * p.v_sh; sn = p.v_sn;
  }
  const int tok0 = kIsQ ? s.tok0_q : s.tok0_k;
  // tile row of the thread's i-th row: E4M3 V (kind 2) gives each thread RPT consecutive
  // tokens, so that four of them form one 32-bit word of the transposed tile; the other kinds
  // interleave the row groups
  auto row_of = [&](int i) { return kind == 2 ? RPT * rg + i : rg + RG * i; };
  uint4 raw[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = r0 + row_of(i);
    raw[i] = (r < len && c0 < d) ? load8_raw<T>(base + (int64_t)(tok0 + r) * sn, c0, d, p.vec16)
                                 : make_uint4(0, 0, 0, 0);
  }
  // smoothed fp32 values of row i (x - mean, one IEEE subtraction; 0 past the end / past d)
  auto row_values = [&](int i, float (&x)[8]) {
    unpack8<T>(raw[i], x);
    const bool live = r0 + row_of(i) < len;
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (live && c0 + j < d) ? __fsub_rn(x[j], mean[j]) : 0.f;
  };
  // the same values in packed arithmetic (x + (-mean) is the same IEEE operation), without the
  // row test: rows past the end read as 0 and give -mean here, and the kinds that use this
  // form zero such rows' maxima and codes themselves; channels past d give 0 - 0
  float nmean[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) nmean[j] = -mean[j];
  auto row_fast = [&](int i, float (&x)[8]) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      unpack2<T>(w[j], x[2 * j], x[2 * j + 1]);
      if (!kIsQ) add2(x[2 * j], x[2 * j + 1], x[2 * j], x[2 * j + 1], nmean[2 * j], nmean[2 * j + 1]);
    }
  };

  if constexpr (kind == 3 || kind == 6) {
    // ---- V: fp16 values (kind 3) or FP4 carriers (kind 6), transposed through shared
    // memory. Element (channel c, token rr) sits at column rr ^ (8 * ((c >> 3) & 15)): whole
    // 16-byte units move, and the 16 threads of a row (one channel octet each) hit different
    // banks.
    __shared__ __align__(16) __half vtile16[128][kTileRows];
    if constexpr (kind == 6) {
      // block maxima of |u| per (16-token block, channel), then each block's scale and rho
      __shared__ unsigned bmax[kTileRows / 16][128];
      __shared__ float brho[kTileRows / 16][128];
      __shared__ __half bscale[kTileRows / 16][128];
      for (int idx = threadIdx.x; idx < (kTileRows / 16) * 128; idx += NT) bmax[idx >> 7][idx & 127] = 0u;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int rr = rg + RG * i;
        float x[8];
        row_values(i, x);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < dp) atomicMax(&bmax[rr >> 4][c0 + j], __float_as_uint(fabsf(__fmul_rn(x[j], rcpv[j]))));
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < (kTileRows / 16) * dp; idx += NT) {
        const int blk = idx / dp, c = idx - blk * dp;
        const Fp4Scale sc = fp4_block_scale(__uint_as_float(bmax[blk][c]));
        brho[blk][c] = sc.rho;
        bscale[blk][c] = __low2half(sc.s2);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int rr = rg + RG * i;
        float x[8];
        row_values(i, x);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const float z0 = __fmul_rn(__fmul_rn(x[j], rcpv[j]), brho[rr >> 4][c0 + j]);
          const float z1 = __fmul_rn(__fmul_rn(x[j + 1], rcpv[j + 1]), brho[rr >> 4][c0 + j + 1]);
          const uint32_t two = fp4_carrier2(z0, z1, __halves2half2(bscale[rr >> 4][c0 + j],
                                                                    bscale[rr >> 4][c0 + j + 1]));
          const __half2 h2 = *reinterpret_cast<const __half2*>(&two);
          vtile16[c0 + j][rr ^ ((vec & 15) << 3)] = __low2half(h2);
          vtile16[c0 + j + 1][rr ^ ((vec & 15) << 3)] = __high2half(h2);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int rr = rg + RG * i;
        float x[8];
        row_values(i, x);
#pragma unroll
        for (int j = 0; j < 8; ++j) vtile16[c0 + j][rr ^ ((vec & 15) << 3)] = __float2half_rn(x[j]);
      }
    }
    __syncthreads();
    const int64_t plane = plane_of(p, b, h, p.hkv);
    const int64_t col0 = (int64_t)s.row0_k + r0;
    const int ncols = (int)min((int64_t)kTileRows, p.vt_pitch - col0);
    __half* vt16 = reinterpret_cast<__half*>(p.vt);
    for (int idx = threadIdx.x; idx < dp * 16; idx += NT) {
      const int c = idx >> 4, u = idx & 15;  // channel, 8-token unit
      if (u * 8 < ncols) {
        const uint4 val = *reinterpret_cast<const uint4*>(&vtile16[c][(u ^ ((c >> 3) & 15)) << 3]);
        *reinterpret_cast<uint4*>(vt16 + (plane * dp + c) * p.vt_pitch + col0 + u * 8) = val;
      }
    }
    return;
  }
  if constexpr (kind == 2) {
    // ---- V: E4M3 codes, transposed through shared memory. Four consecutive tokens of a
    // channel form one 32-bit word; word w of channel row c sits in 16-byte chunk
    // (w / 4) ^ ((c / 8) & 7), so the warp's stores spread over the banks.
    __shared__ __align__(16) uint8_t vtile[128][kTileRows];
#pragma unroll
    for (int qd = 0; qd < RPT / 4; ++qd) {
      uint32_t cw[4][4];  // [token][channel pair]: E4M3 bytes of channels 2j (low), 2j + 1
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = 4 * qd + t;
        float x[8], y[8];
        row_fast(i, x);
#pragma unroll
        for (int j = 0; j < 8; j += 2) mul2(y[j], y[j + 1], x[j], x[j + 1], rcpv[j], rcpv[j + 1]);
        const bool live = r0 + row_of(i) < len;
#pragma unroll
        for (int j = 0; j < 4; ++j) cw[t][j] = live ? pack_e4m3x2(y[2 * j], y[2 * j + 1]) : 0u;
      }
      const int tw = (RPT / 4) * rg + qd;                      // token word within the row
      const int byte = (((tw >> 2) ^ (vec & 7)) << 4) + ((tw & 3) << 2);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (c0 + 2 * j < dp) {
          const uint32_t lo01 = __byte_perm(cw[0][j], cw[1][j], 0x5410);  // t0c0 t0c1 t1c0 t1c1
          const uint32_t lo23 = __byte_perm(cw[2][j], cw[3][j], 0x5410);  // t2c0 t2c1 t3c0 t3c1
          *reinterpret_cast<uint32_t*>(&vtile[c0 + 2 * j][byte]) = __byte_perm(lo01, lo23, 0x6420);
          *reinterpret_cast<uint32_t*>(&vtile[c0 + 2 * j + 1][byte]) = __byte_perm(lo01, lo23, 0x7531);
        }
      }
    }
    __syncthreads();
    // row c of the transposed tile = bytes [r0, r0 + 128) of channel c; write the bytes that
    // exist in this plane's pitch (a multiple of 16), 16 bytes per thread
    const int64_t plane = plane_of(p, b, h, p.hkv);
    const int64_t col0 = (int64_t)s.row0_k + r0;
    const int ncols = (int)min((int64_t)kTileRows, p.vt_pitch - col0);
    for (int idx = threadIdx.x; idx < dp * 8; idx += NT) {
      const int c = idx >> 3, ch = (idx & 7) * 16;
      if (ch < ncols) {
        uint4 val = *reinterpret_cast<const uint4*>(&vtile[c][ch ^ (((c >> 3) & 7) << 4)]);
        *reinterpret_cast<uint4*>(p.vt + (plane * dp + c) * p.vt_pitch + col0 + ch) = val;
      }
    }
    return;
  }

  // ---- Q / K: INT8 codes (kinds 0, 1) or FP4 carriers (kinds 4, 5) per token group
  constexpr bool kFp4 = kind >= 4;
  constexpr float kRange = kFp4 ? 448.0f : 127.0f;  // the group's absmax maps onto this
  const int gs = kIsQ ? p.gq : p.gk;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    float x[8];
    row_fast(i, x);
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(x[j]));
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (vec == 0) rowmax[rg + RG * i] = r0 + rg + RG * i < len ? a : 0.f;  // past the end: 0
  }
  __syncthreads();
  const int64_t plane = plane_of(p, b, h, kIsQ ? p.hq : p.hkv);
  const int row0 = kIsQ ? s.row0_q : s.row0_k;
  {
    // group absmax: warps 0-3 each own 32 consecutive rows; groups of <= 32 rows reduce with
    // shuffles, groups of 64 / 128 rows combine the per-warp maxima
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float wmax[4];
    float a = 0.f;
    if (warp < 4) {
      a = rowmax[warp * 32 + lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1)
        if (off < gs) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
      if (lane == 0) wmax[warp] = a;
    }
    __syncthreads();
    if (warp < 4 && gs > 32) {
      const int w0 = (warp * 32 / gs) * (gs / 32);
      a = wmax[w0];
      for (int w = 1; w < gs / 32; ++w) a = fmaxf(a, wmax[w0 + w]);
    }
    const int r = warp * 32 + lane;  // row of this lane (warps 0-3)
    if (warp < 4 && r % gs == 0) {
      const int g = r / gs;
      grcp[g] = a > 0.f ? __fdiv_rn(kRange, a) : 0.f;
      if (r0 + r < len) {
        float* sc = kIsQ ? p.sq : p.sk;
        const int64_t pp = kIsQ ? p.sq_pp : p.sk_pp;
        sc[plane * pp + (row0 + r0) / gs + g] = a > 0.f ? __fdiv_rn(a, kRange) : 0.f;
      }
    }
  }
  __syncthreads();
  __half* codes = kIsQ ? p.qc : p.kc;
  const int64_t rows_pp = kIsQ ? p.q_rows : p.k_rows;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int rr = rg + RG * i;
    const int r = r0 + rr;
    const float rc = grcp[rr / gs];
    float x[8];
    row_fast(i, x);
    __align__(16) __half2 hv[4];
    if constexpr (kFp4) {
      // u = fl32(x * r); the 16-channel block of this row spans this thread and its
      // neighbour (vec ^ 1)
      float u[8], m = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        u[j] = __fmul_rn(x[j], rc);
        m = fmaxf(m, fabsf(u[j]));
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      const Fp4Scale sc = fp4_block_scale(m);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const uint32_t two = fp4_carrier2(__fmul_rn(u[j], sc.rho), __fmul_rn(u[j + 1], sc.rho), sc.s2);
        hv[j / 2] = *reinterpret_cast<const __half2*>(&two);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        // rint_even(fl32(x * r)) via the rounding constant. Scalar IEEE operations on purpose:
        // the compiler may fuse a packed multiply and the packed add after it into one packed
        // fma, whose single rounding moves products that round to a tie (63.5) in fp32. No
        // clamp is needed: r = fl32(127 / absmax) exceeds 127 / absmax by at most a relative
        // 2^-24, so |fl32(x * r)| <= 127 + 2^-17 and its rounding is at most 127.
        const float c0 = __fsub_rn(__fadd_rn(__fmul_rn(x[j], rc), kRoundMagic), kRoundMagic);
        const float c1 = __fsub_rn(__fadd_rn(__fmul_rn(x[j + 1], rc), kRoundMagic), kRoundMagic);
        hv[j / 2] = __floats2half2_rn(c0, c1);  // exact: integers of magnitude <= 127
      }
    }
    if (r >= len) {
#pragma unroll
      for (int j = 0; j < 4; ++j) hv[j] = __half2{};  // rows past the end are stored as zeros
    }
    if (c0 < dp && r < stored)
      *reinterpret_cast<uint4*>(codes + (plane * rows_pp + row0 + r) * dp + c0) =
          *reinterpret_cast<const uint4*>(hv);
    if (want_qkc) {
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) dot = fmaf(x[j], kmean_q[j], dot);
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (vec == 0 && r < len) p.qkc[plane * p.q_rows + row0 + r] = dot;
    }
  }
}

// Q, K and V quantisation in one launch. Grid: (128-token tiles of the longest sequence,
// Hq + 2 Hkv, batch): blockIdx.y selects a Q head, then a K head, then a V head.
// VM: 0 = FP8 V, 1 = fp16 V (FP16 P·V variant), 2 = FP4 microscaled Q, K and V.
template <typename T, int TPR, int VM, int NT>
__global__ void __launch_bounds__(NT, NT == 512 ? 2 : (TPR == 8 ? 4 : 3)) quant_kernel(Problem p) {
  pdl_trigger();
  pdl_wait();  // the finalisation's means and scales
  const int y = blockIdx.y;
  if (y < p.hq) quant_block<T, VM == 2 ? 4 : 0, TPR, NT>(p, blockIdx.x, y, blockIdx.z);
  else if (y < p.hq + p.hkv) quant_block<T, VM == 2 ? 5 : 1, TPR, NT>(p, blockIdx.x, y - p.hq, blockIdx.z);
  else quant_block<T, VM == 0 ? 2 : (VM == 1 ? 3 : 6), TPR, NT>(p, blockIdx.x, y - p.hq - p.hkv, blockIdx.z);
}

// ------------------------------------------------------------------------------------------
// Export of the quantised state in canonical layouts (test hook).
__global__ void export_codes_kernel(const __half* codes, int64_t rows_pp, int dp, int d,
                                    int planes, int n, int8_t* out) {
  const int64_t total = (int64_t)planes * n * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % d);
    const int64_t r = (i / d) % n, pl = i / ((int64_t)d * n);
    out[i] = static_cast<int8_t>(__half2int_rn(codes[(pl * rows_pp + r) * dp + c]));
  }
}
__global__ void export_vt_kernel(const uint8_t* vt, int64_t pitch, int dp, int d, int planes,
                                 int n, uint8_t* out) {
  const int64_t total = (int64_t)planes * n * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % d);
    const int64_t r = (i / d) % n, pl = i / ((int64_t)d * n);
    out[i] = vt[(pl * dp + c) * pitch + r];
  }
}
__global__ void export_fp16_kernel(const __half* codes, int64_t rows_pp, int dp, int d,
                                   int planes, int n, uint16_t* out) {
  const int64_t total = (int64_t)planes * n * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % d);
    const int64_t r = (i / d) % n, pl = i / ((int64_t)d * n);
    out[i] = __half_as_ushort(codes[(pl * rows_pp + r) * dp + c]);
  }
}
__global__ void export_vt16_kernel(const __half* vt, int64_t pitch, int dp, int d, int planes,
                                   int n, uint16_t* out) {
  const int64_t total = (int64_t)planes * n * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % d);
    const int64_t r = (i / d) % n, pl = i / ((int64_t)d * n);
    out[i] = __half_as_ushort(vt[(pl * dp + c) * pitch + r]);
  }
}
__global__ void e2m1_kernel(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint16_t c;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(c)
        : "f"(0.f), "f"(x[i]));
    out[i] = static_cast<uint8_t>(c & 0xF);
  }
}
__global__ void e4m3_kernel(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = static_cast<uint8_t>(pack_e4m3x2(x[i], 0.f) & 0xFF);
}

// ------------------------------------------------------------------------------------------
// Host launchers (all on the caller's stream).
cudaError_t launch_varlen_setup(const Problem& p, cudaStream_t st) {
  varlen_setup_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
static void launch_kv_stats_t(const Problem& p, dim3 grid, int nb, cudaStream_t st) {
  if (p.dp == 64) kv_stats_kernel<T, 8><<<grid, 256, 0, st>>>(p, nb);
  else kv_stats_kernel<T, 16><<<grid, 256, 0, st>>>(p, nb);
}

cudaError_t launch_kv_stats(const Problem& p, int max_len_k, cudaStream_t st) {
  // tokens per batch (4 rows per thread); batches per block: 4 where that still leaves twelve
  // blocks for each of the 152 SMs, else fewer
  const int batch_rows = stats_chunk(p.dp);
  const int tensors = p.smooth_k ? 2 : 1;
  int nb = 4;
  auto blocks = [&](int n) {
    return (int64_t)((max_len_k + batch_rows * n - 1) / (batch_rows * n)) * p.hkv * p.batch * tensors;
  };
  while (nb > 1 && blocks(nb) < 152 * 12) nb >>= 1;
  const dim3 grid((max_len_k + batch_rows * nb - 1) / (batch_rows * nb), p.hkv, p.batch * tensors);
  if (p.dtype == 0) launch_kv_stats_t<__half>(p, grid, nb, st);
  else launch_kv_stats_t<__nv_bfloat16>(p, grid, nb, st);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const Problem& p, int n_stats, cudaStream_t st) {
  const cudaError_t e = launch_pdl(kv_finalize_kernel, dim3((n_stats + 255) / 256), dim3(256), 0, st, p, n_stats);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_quant_t(const Problem& p, int max_len_q, int max_len_k, cudaStream_t st) {
  const int len = max_len_q > max_len_k ? max_len_q : max_len_k;
  const dim3 grid((len + kTileRows - 1) / kTileRows, p.hq + 2 * p.hkv, p.batch);
  const int vm = p.fp4 ? 2 : (p.pv16 ? 1 : 0);
  if (p.dp == 64) {
    return vm == 2 ? launch_pdl(quant_kernel<T, 8, 2, 256>, grid, dim3(256), 0, st, p)
         : vm == 1 ? launch_pdl(quant_kernel<T, 8, 1, 256>, grid, dim3(256), 0, st, p)
                   : launch_pdl(quant_kernel<T, 8, 0, 256>, grid, dim3(256), 0, st, p);
  } else if (!p.varlen) {
    return vm == 2 ? launch_pdl(quant_kernel<T, 16, 2, 512>, grid, dim3(512), 0, st, p)
         : vm == 1 ? launch_pdl(quant_kernel<T, 16, 1, 512>, grid, dim3(512), 0, st, p)
                   : launch_pdl(quant_kernel<T, 16, 0, 512>, grid, dim3(512), 0, st, p);
  } else {
    // the FP4 variant has no varlen entry point
    return vm == 1 ? launch_pdl(quant_kernel<T, 16, 1, 256>, grid, dim3(256), 0, st, p)
                   : launch_pdl(quant_kernel<T, 16, 0, 256>, grid, dim3(256), 0, st, p);
  }
}

cudaError_t launch_quant(const Problem& p, int max_len_q, int max_len_k, cudaStream_t st) {
  const cudaError_t e = p.dtype == 0 ? launch_quant_t<__half>(p, max_len_q, max_len_k, st)
                                     : launch_quant_t<__nv_bfloat16>(p, max_len_q, max_len_k, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_export_codes(const __half* codes, int64_t rows_pp, int dp, int d, int planes,
                                int n, int8_t* out, cudaStream_t st) {
  export_codes_kernel<<<1024, 256, 0, st>>>(codes, rows_pp, dp, d, planes, n, out);
  return cudaGetLastError();
}

cudaError_t launch_export_vt(const uint8_t* vt, int64_t pitch, int dp, int d, int planes, int n,
                             uint8_t* out, cudaStream_t st) {
  export_vt_kernel<<<1024, 256, 0, st>>>(vt, pitch, dp, d, planes, n, out);
  return cudaGetLastError();
}

cudaError_t launch_e2m1(const float* x, uint8_t* out, int64_t n, cudaStream_t st) {
  e2m1_kernel<<<1024, 256, 0, st>>>(x, out, n);
  return cudaGetLastError();
}

cudaError_t launch_export_fp16(const __half* codes, int64_t rows_pp, int dp, int d, int planes,
                               int n, uint16_t* out, cudaStream_t st) {
  export_fp16_kernel<<<1024, 256, 0, st>>>(codes, rows_pp, dp, d, planes, n, out);
  return cudaGetLastError();
}

cudaError_t launch_export_vt16(const __half* vt, int64_t pitch, int dp, int d, int planes, int n,
                               uint16_t* out, cudaStream_t st) {
  export_vt16_kernel<<<1024, 256, 0, st>>>(vt, pitch, dp, d, planes, n, out);
  return cudaGetLastError();
}

cudaError_t launch_e4m3(const float* x, uint8_t* out, int64_t n, cudaStream_t st) {
  e4m3_kernel<<<1024, 256, 0, st>>>(x, out, n);
  return cudaGetLastError();
}

}  // namespace sage
