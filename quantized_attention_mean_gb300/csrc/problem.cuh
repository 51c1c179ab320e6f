// Problem descriptor shared by the host API and the kernels, the workspace layout, and the
// small device helpers (input loads, per-sequence geometry, FP8 packing, error recording).
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace sage {

constexpr int kTileRows = 128;   // query rows per attention tile, tokens per quantisation tile
constexpr int kTileKeys = 128;   // keys per attention KV tile
// tokens per batch of the K/V statistics pass (4 rows per thread, dp/8 threads per row)
__host__ __device__ constexpr int stats_chunk(int dp) { return 8192 / dp; }

// Device-side status codes (mirror sage_status in include/sageattn.h).
enum DevStatus : int { kDevOk = 0, kDevRange = 7, kDevTimeout = 9, kDevSeqlens = 12 };

// Everything the kernels need. Strides are in elements; offset of (seq b, token t, head h)
// in an input/output tensor is b*s_b + (tok0(b) + t)*s_n + h*s_h, where tok0 = 0 for dense
// problems and cu_seqlens[b] for varlen (whose s_b is 0).
struct Problem {
  int batch, hq, hkv, d, dp;       // dp: padded head_dim (64 or 128)
  int nq, nk;                      // dense: sequence lengths; varlen: max lengths
  int varlen, dtype, is_causal, return_lse, smooth_k, smooth_v;
  int gq, gk, lgk;                 // token-group sizes of Q and K scales; lgk = log2(gk)
  int vec16;                       // inputs allow 16-byte vector loads
  int pv16;                        // P·V on fp16 operands: V^T stored as fp16, P in fp16
  int fp4;                         // FP4 microscaled variant (with pv16): Q, K, V, P carried
                                   // as E2M1 code x E4M3 block scale in fp16
  int pair_major;                  // attention CTAs ordered pairs-fastest (see api.cu)
  float sm_scale;
  float range_limit;               // smallest float >= 2^38 / N (dense only; varlen per seq)
  const void* q; int64_t q_sb, q_sh, q_sn;
  const void* k; int64_t k_sb, k_sh, k_sn;
  const void* v; int64_t v_sb, v_sh, v_sn;
  void* o;       int64_t o_sb, o_sh, o_sn;
  float* lse;                      // dense [B,Hq,Nq]; varlen [Hq,total_q]
  int64_t lse_plane;               // varlen: total_q
  const int* cu_q; const int* cu_k;
  int total_q, total_k;
  // workspace
  int* err;
  long long* ksum; long long* vsum;                           // [batch*hkv*d]
  unsigned* vmin; unsigned* vmax;  // [batch*hkv*d] order-preserving codes, zero = empty
  float* kmean; float* vmean; float* vscale; float* vrcp;     // [batch*hkv*d]
  __half* qc; __half* kc; uint8_t* vt;  // codes; vt holds E4M3 bytes or (pv16) fp16 V^T
  float* sq; float* sk; float* qkc;                           // scales, LSE correction
  int* seqinfo;                    // varlen: [kSiRows][batch] per-sequence geometry + LPT order
  int64_t q_rows, k_rows;          // rows per plane in qc / kc (dense: nq / nk)
  int64_t vt_pitch;                // elements per channel row of vt (1 or 2 bytes each)
  int64_t sq_pp, sk_pp;            // scale groups per plane
  int32_t* dbg_scores;             // optional exact-score dump [B,Hq,Nq,Nk]
  int dbg_stall;                   // test hook: the producer issues no K/V loads
  long long* dbg_trace;            // optional event clocks of CTA (0,0,0): [4 roles][64 tiles][8]
};

constexpr int kTraceTiles = 64, kTraceEvents = 8;

struct Seq {
  int tok0_q, len_q, row0_q, tok0_k, len_k, row0_k;
};

// varlen seqinfo rows (each of length batch)
enum { kSiTok0Q = 0, kSiLenQ, kSiRow0Q, kSiTok0K, kSiLenK, kSiRow0K, kSiOrder, kSiRows };

__device__ __forceinline__ Seq get_seq(const Problem& p, int b) {
  Seq s;
  if (!p.varlen) {
    s.tok0_q = 0; s.len_q = p.nq; s.row0_q = 0;
    s.tok0_k = 0; s.len_k = p.nk; s.row0_k = 0;
  } else {
    const int* si = p.seqinfo;
    const int B = p.batch;
    s.tok0_q = si[kSiTok0Q * B + b]; s.len_q = si[kSiLenQ * B + b]; s.row0_q = si[kSiRow0Q * B + b];
    s.tok0_k = si[kSiTok0K * B + b]; s.len_k = si[kSiLenK * B + b]; s.row0_k = si[kSiRow0K * B + b];
  }
  return s;
}

// Plane index of (sequence b, head h) in the code/scale arrays.
__device__ __forceinline__ int64_t plane_of(const Problem& p, int b, int h, int heads) {
  return p.varlen ? (int64_t)h : (int64_t)b * heads + h;
}

__device__ __forceinline__ void record_error(int* err, int code) { atomicCAS(err, 0, code); }

// Programmatic dependent launch (no-ops for kernels launched without it): wait until the
// previous kernel in the stream has completed and its writes are visible; let the next
// kernel begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Loads channels [c0, c0+8) of one row; channels >= d read as 0.
template <typename T>
__device__ __forceinline__ void load8(const T* row, int c0, int d, int vec16, float (&x)[8]) {
  if (vec16 && c0 + 8 <= d) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(row + c0));
    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = to_f32<T>(h[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = (c0 + i < d) ? to_f32<T>(row[c0 + i]) : 0.0f;
  }
}

// Raw 16-byte load of channels [c0, c0+8) of one row (channels >= d read as 0).
template <typename T>
__device__ __forceinline__ uint4 load8_raw(const T* row, int c0, int d, int vec16) {
  if (vec16 && c0 + 8 <= d) return __ldg(reinterpret_cast<const uint4*>(row + c0));
  __align__(16) T h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = (c0 + i < d) ? row[c0 + i] : T(0.0f);
  return *reinterpret_cast<const uint4*>(h);
}
template <typename T>
__device__ __forceinline__ void unpack8(uint4 u, float (&x)[8]) {
  const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = to_f32<T>(h[i]);
}

// Two floats -> two E4M3 bytes (RNE, saturate to +-448): byte 0 = lo, byte 1 = hi.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- FP4 microscaling (pwwt.cn guide §5.5, SageAttention3 "FP4 microscaling"): E2M1
// elements, one E4M3 scale per block of 16 along the dot-product dimension. A block's scale
// s is its largest mapped magnitude rounded to E4M3; each element is coded as
// e2m1(fl32(u · fl32(6 / s))) and enters the tensor cores as its carrier code · s, which fp16
// holds exactly (at most 5 significant bits, between 2^-10 and 2688).

// E4M3 block scale of a block maximum m >= 0: its value as an fp16 pair (both halves) and
// rho = fl32(6 / s) (0 when s = 0).
struct Fp4Scale {
  __half2 s2;
  float rho;
};
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t codes16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(codes16)));
  return *reinterpret_cast<__half2*>(&h);
}
__device__ __forceinline__ Fp4Scale fp4_block_scale(float m) {
  Fp4Scale r;
  r.s2 = e4m3x2_to_half2(pack_e4m3x2(m, m));
  const float s = __low2float(r.s2);
  r.rho = s > 0.f ? __fdiv_rn(6.0f, s) : 0.f;
  return r;
}
// Two already scaled values z = fl32(u · rho) to their E2M1 codes (RNE, saturating at ±6) and
// back as an fp16 pair, times the pair's block scales s2: the two carriers, z0 in the low half.
__device__ __forceinline__ uint32_t fp4_carrier2(float z0, float z1, __half2 s2) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h)
      : "f"(z1), "f"(z0));
  const __half2 c = __hmul2(*reinterpret_cast<const __half2*>(&h), s2);  // exact
  return *reinterpret_cast<const uint32_t*>(&c);
}

// Order-preserving float -> unsigned map (a larger float has a larger code, and every
// non-NaN float's code is above 0), so a zero-filled buffer is an empty atomicMax
// accumulator. The minimum is kept as the maximum of the complemented code.
__device__ __forceinline__ unsigned ordered_code(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_decode(unsigned c) {
  return __uint_as_float((c & 0x80000000u) ? (c & 0x7FFFFFFFu) : ~c);
}

// Adding 1.5 * 2^23 rounds an fp32 value v with |v| < 2^22 to an integer (ties to even, the
// IEEE default), which the sum then holds in its low mantissa bits: the integer is
// bits(v + 1.5 * 2^23) - bits(1.5 * 2^23). This replaces float -> int conversions, which run on
// a slow pipe (fp32 -> int64 at ~2 per clock per SM on this GPU).
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kRoundMagicBits = 0x4B400000;

// x * 2^24 split exactly into hi * 2^20 + lo with hi = round(x * 16), lo = (x * 16 - hi) * 2^20.
// Exact whenever x * 2^24 is an integer and |x| < 2^18 (every fp16 value; bf16 values of
// magnitude >= 2^-17 or 0): then r = x * 16 - hi is exact and r * 2^20 is an integer < 2^19.
// The two words are returned with the rounding constant's bit pattern still in them (hi + and
// lo + kRoundMagicBits): summing them modulo 2^32 and subtracting n * kRoundMagicBits once
// gives the sums of n (hi, lo) pairs exactly, as long as those true sums fit in an int32.
__device__ __forceinline__ void fixed_split_biased(float x, unsigned& hi, unsigned& lo) {
  const float t1 = __fmaf_rn(x, 16.0f, kRoundMagic);
  hi = __float_as_uint(t1);
  const float r = __fmaf_rn(x, 16.0f, -__fsub_rn(t1, kRoundMagic));
  lo = __float_as_uint(__fmaf_rn(r, 1048576.0f, kRoundMagic));
}

template <typename T>
__device__ __forceinline__ bool fixed_split_exact(float x) {
  if (std::is_same<T, __half>::value) return true;  // |x| <= 65504, multiples of 2^-24
  const float a = fabsf(x);
  return a < 262144.0f && (a >= 7.62939453125e-06f || a == 0.0f);
}

// Exact, order-free mean from the fixed-point sum: fl32(fl64(fl64(S) * 2^-24 / n)).
__device__ __forceinline__ float fixed_point_mean(long long s, int n) {
  double m = __dmul_rn(__ll2double_rn(s), 5.9604644775390625e-08);  // * 2^-24, exact
  return __double2float_rn(__ddiv_rn(m, (double)n));
}

}  // namespace sage
