// Stage 3 of the method (pwwt.cn "SageAttention deployment pitfalls guide" §1, §4.1, §4.2;
// pnsm.cn "SageAttention on AMD 9070 XT without the HIP SDK" §2: FlashAttention-style
// tiling with a quantisation layer): a fused, warp-specialised attention kernel for sm_103a.
//
// One CTA owns two 128-row query tiles (A and B) of one (sequence, query head) and walks the
// KV tiles of 128 keys:
//   warp 8      TMA producer: Q tiles once, then K tiles (integer-valued fp16 codes) and
//               V^T tiles (E4M3) through a ring of shared-memory stages;
//   warps 9, 10 issue the MMAs from one elected thread each, warp 9 for query tile A (and
//               allocates tensor memory), warp 10 for tile B:
//               S = Q8 . K8^T  (tcgen05 kind::f16 on the INT8 codes: every product and partial
//                               sum is an integer below 2^24, so the fp32 accumulator holds
//                               the exact INT32 score),
//               O += P~ . V~   (tcgen05 kind::f8f6f4, E4M3 x E4M3 -> fp32 in tensor memory);
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: one thread per query row
//               reads its S row from tensor memory, dequantises (s_q . s_k . sm_scale),
//               masks, keeps the running max / sum, writes P~ = e4m3(2^(x - m) . sigma_P) to
//               shared memory, rescales its O row in tensor memory when the max grows, and
//               finally writes O = acc . s_v / l + v_mean and the LSE.
// The two tiles ping-pong: while one tile's softmax runs, the tensor core computes the other
// tile's scores, and each tile's next S is computed while its current softmax still runs.
// Tensor memory at head_dim 128: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512); a
// tile's issuer starts its next QK^T as soon as the softmax holds S in registers (s_free),
// and its P.V once P is written and O rescaled (o_ready). At head_dim 64 three S buffers
// [0,384) rotate over the tiles in issue order (A_0, B_0, A_1, B_1, ...; item n in buffer
// n % 3), O_A [384,448), O_B [448,512): once a tile's softmax has published P (p_full), its
// issuer issues the tile's P.V and then the scores three items ahead into the freed buffer.
// With one issuer per tile, one issuer's barrier waits and commits overlap the other's MMAs.
//
// Variants (template argument PV): 0 = E4M3 P and V on kind::f8f6f4; 1 = the FP16 P·V
// variant (P and V' in fp16 on kind::f16); 2 = the FP4 microscaled variant (pwwt.cn guide
// §5.5): Q, K, V arrive as fp16 carriers of E2M1 codes x E4M3 block scales, and the softmax
// quantises P the same way per 16 keys (scale = e4m3 of the block's largest 448 p,
// codes = e2m1(448 p . fl32(6 / scale))); both products run on kind::f16, where every carrier
// product is exact.
//
// Every wait is bounded; a timeout records SAGE_ERR_TIMEOUT and all roles exit cleanly.
#include "launch.h"
#include "problem.cuh"
#include "sm103_ptx.cuh"

namespace sage {

// 12 warps = 3 warpgroups: softmax A (warps 0-3), softmax B (4-7), and a control warpgroup
// (warp 8 TMA, warp 9 tile A's MMAs + TMEM allocation, warp 10 tile B's MMAs, warp 11
// idle). Launched at 168 registers
// per thread (the per-sub-partition limit with 3 warps each); the control warpgroup drops to
// 56 and the softmax warpgroups rise to 224: 2*128*224 + 128*56 = 12*32*168.
constexpr int kAttnThreads = 384;
constexpr uint32_t kRegsSoftmax = 224, kRegsControl = 56;
constexpr float kLog2e = 1.4426950408889634f;

// PV16: the FP16 P·V variant (P and V' in fp16, P·V on kind::f16); otherwise E4M3 P and V.
template <int DP, bool PV16 = false>
struct AttnCfg {
  static constexpr int kChunks = DP / 64;                       // 128-byte K-chunks of a row
  static constexpr int kQTileBytes = kTileRows * DP * 2;        // fp16 codes
  static constexpr int kKTileBytes = kTileKeys * DP * 2;
  static constexpr int kVTileBytes = DP * kTileKeys * (PV16 ? 2 : 1);    // V^T, E4M3 or fp16
  static constexpr int kPTileBytes = kTileRows * kTileKeys * (PV16 ? 2 : 1);  // E4M3 or fp16
  static constexpr int kKStages = DP == 128 ? 2 : 4;
  static constexpr int kVStages = DP == 128 ? (PV16 ? 1 : 2) : 4;
  // P buffers per query tile: with two, the softmax writes P_j while P.V of tile j - 1 may
  // still be reading P_{j-1} (the FP16 P·V variant has room for one)
  static constexpr int kPBufs = PV16 ? 1 : 2;
  // S buffers in tensor memory: at head_dim 64 three 128-column buffers serve the two query
  // tiles in rotation (item n = tile j of query tile x, n = j * tiles + x, uses buffer n % 3),
  // so a tile's next scores are computed while its softmax still runs; at 128 the two O
  // accumulators leave room for one buffer per query tile
  static constexpr int kSBufs = DP == 64 ? 3 : 2;
  static constexpr uint32_t kTmemO = kSBufs * 128;  // O of query tile x at kTmemO + x * DP
  // with the rotating S buffers a K tile is needed a tile ahead of its V tile anyway: K and V
  // of one tile share a stage, one full barrier (k_full) and one release (k_empty)
  static constexpr bool kKVShared = kSBufs == 3;
  static_assert(kTmemO + 2 * DP <= 512, "tensor memory columns");
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kKTileBytes;
  static constexpr int kOffP = kOffV + kVStages * kVTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBufs * kPTileBytes;
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + kSBufs + 6 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRho = kOffMisc + 64;  // FP4: fl32(6 / s) per E4M3 code s (128)
  static constexpr int kBytes = kOffRho + 128 * 4;
  // one CTA per SM (the kernel allocates all 512 tensor-memory columns)
  static constexpr int kSmem = (kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024);
  static_assert(kBytes + 1024 <= 232448, "shared memory budget");
  // shared stages: the MMA issuer asks for K_{j+3} (the scores three items ahead, one query
  // tile) before it issues P_j V_j, whose completion releases the stage of tile j + 3 - stages;
  // so a single query tile needs more than three stages
  static_assert(!kKVShared || (kKStages == kVStages && kKStages >= 4), "shared K / V stages");
};

// Instruction descriptors: M = 128 rows, fp32 accumulate, K-major operands.
__host__ __device__ constexpr uint32_t idesc_qk() { return make_idesc(1, 0, 0, 128, 128); }
template <int DP>
__host__ __device__ constexpr uint32_t idesc_pv() { return make_idesc(1, 0, 0, 128, DP); }


__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four MMAs of one kind into d from one elected lane of a converged warp: operands (a_k, b_k),
// k = 0..3, the first accumulating when acc0 != 0 and the others always.
template <bool F8>
__device__ __forceinline__ void mma4_warp(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2, uint64_t a3,
                                          uint64_t b0, uint64_t b1, uint64_t b2, uint64_t b3,
                                          uint32_t idesc, uint32_t acc0) {
  if constexpr (F8) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 q, %10, %10;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %5, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %6, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %7, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %8, %9, q;\n\t}" ::"r"(d),
        "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(acc0)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 q, %10, %10;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, q;\n\t}" ::"r"(d),
        "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(acc0)
        : "memory");
  }
}

// a[idx] for a runtime idx in [0, 32) without indexing a register array.
__device__ __forceinline__ uint32_t pick32(const uint32_t (&a)[32], int idx) {
  uint32_t v = a[0];
#pragma unroll
  for (int g = 1; g < 32; ++g) v = idx == g ? a[g] : v;
  return v;
}

// Two output values as fp16 (dtype 0) or bf16 bits, the first in the low half.
__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, int dtype) {
  if (dtype == 0) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// V scales and means of the channels [c0, c0 + 32) as 16-byte loads, 8-channel groups at or
// past d left zero (d % 8 == 0; the rows start 32-byte aligned).
__device__ __forceinline__ void load_chunk_scales(const float* vsc, const float* vmn, int c0, int d,
                                                  float4 (&cs)[8], float4 (&cm)[8]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (c0 + q * 8 < d) {
      const float4* s4 = reinterpret_cast<const float4*>(vsc + c0 + q * 8);
      const float4* m4 = reinterpret_cast<const float4*>(vmn + c0 + q * 8);
      cs[2 * q] = __ldg(s4);
      cs[2 * q + 1] = __ldg(s4 + 1);
      cm[2 * q] = __ldg(m4);
      cm[2 * q + 1] = __ldg(m4 + 1);
    } else {
      cs[2 * q] = cs[2 * q + 1] = cm[2 * q] = cm[2 * q + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// a[idx] for a runtime idx in [0, 8) without indexing a register array.
__device__ __forceinline__ float pick8(const float (&a)[8], int idx) {
  float v = a[0];
#pragma unroll
  for (int g = 1; g < 8; ++g) v = idx == g ? a[g] : v;
  return v;
}

// ---- rarely taken softmax paths, kept out of line so the hot loop stays small in the
// instruction cache. They re-read S from tensor memory 32 columns at a time.
struct Mult8 {
  float v[8];
};

// Test hook: the integer scores of one row of the tile as read from tensor memory.
__device__ __noinline__ void dump_scores_row(uint32_t tS, bool row_valid, int32_t* dst, int ncols) {
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t t[32];
    tmem_ld32(tS + ch * 32, t);
    tmem_wait_ld(t);
    if (row_valid) {
#pragma unroll
      for (int u = 0; u < 32; ++u)
        if (ch * 32 + u < ncols) dst[ch * 32 + u] = __float2int_rn(__uint_as_float(t[u]));
    }
  }
}

// Max over the keys [0, limit) of the tile of S * c (c per 16-key sub-group).
__device__ __noinline__ float masked_tile_max(uint32_t tS, int limit, Mult8 cg) {
  float tile_max = __int_as_float(0xff800000);
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t t[32];
    tmem_ld32(tS + ch * 32, t);
    tmem_wait_ld(t);
    const float c0 = pick8(cg.v, 2 * ch), c1 = pick8(cg.v, 2 * ch + 1);
#pragma unroll
    for (int u = 0; u < 32; ++u)
      if (ch * 32 + u < limit) tile_max = fmaxf(tile_max, __uint_as_float(t[u]) * (u < 16 ? c0 : c1));
  }
  return tile_max;
}

// Stores the P values of one 16-key group g of row r (w: E4M3 bytes or fp16 pairs) into the
// row's P buffer: 128-byte swizzled K-major rows, E4M3 one 16-byte unit per group, fp16 two
// units per group with 64 keys per 128-row chunk.
template <bool PV16>
__device__ __forceinline__ void store_p_group(uint8_t* my_p, int r, int g, const uint32_t (&w)[PV16 ? 8 : 4]) {
  if constexpr (PV16) {
    uint8_t* chunk = my_p + (g >> 2) * (kTileRows * 128);
    const int u0 = (g & 3) * 2;
    *reinterpret_cast<uint4*>(chunk + ((u0 ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(chunk + (((u0 + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
    *reinterpret_cast<uint4*>(my_p + ((g ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
// Two P values in the P buffer's format: E4M3 (bits 0-15 used) or an fp16 pair.
template <bool PV16>
__device__ __forceinline__ uint32_t pack_p2(float lo, float hi) {
  if constexpr (PV16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    return pack_e4m3x2(lo, hi);
  }
}

// Four values as E4M3 bytes of one word, the first in the lowest byte (RNE, saturating).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t w;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return w;
}

// Largest of 16 values.
__device__ __forceinline__ float max16(const float (&e)[16]) {
  float m = max3(e[0], e[1], e[2]);
#pragma unroll
  for (int u = 3; u < 15; u += 2) m = max3(m, e[u], e[u + 1]);
  return fmaxf(m, e[15]);
}

// FP4 carriers of one 16-key group of y = 448 p values (y >= 0): the block scale is the
// E4M3 rounding of the group's largest y, the codes e2m1(fl32(y . fl32(6 / scale))); rho_tab
// holds fl32(6 / s) for every non-negative E4M3 code s.
__device__ __forceinline__ void fp4_p_group(const float (&e)[16], float emax, const float* rho_tab,
                                            uint32_t (&w)[8]) {
  const uint32_t code = pack_e4m3x2(emax, 0.f);
  const __half2 s2 = e4m3x2_to_half2((code & 0xffu) * 0x101u);
  const float rho = rho_tab[code & 0x7fu];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float z0, z1;
    mul2(z0, z1, e[2 * k], e[2 * k + 1], rho, rho);
    w[k] = fp4_carrier2(z0, z1, s2);
  }
}

// P~ = fmt(2^(S*c + bias)) for keys [0, limit) (0 beyond), written to the row's swizzled
// P buffer; returns the row sum of the unquantised values.
template <int PV>
__device__ __noinline__ float masked_tile_exp(uint32_t tS, int limit, Mult8 cg, float bias,
                                              uint8_t* my_p, int r, const float* rho_tab) {
  constexpr bool PV16 = PV != 0;
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t t[32];
    tmem_ld32(tS + ch * 32, t);
    tmem_wait_ld(t);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float cgc = pick8(cg.v, 2 * ch + half);
      uint32_t w[PV16 ? 8 : 4];
      if constexpr (PV == 2) {
        float e[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int uu = half * 16 + u;
          e[u] = ch * 32 + uu < limit ? ex2(fmaf(__uint_as_float(t[uu]), cgc, bias)) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; u += 4) {
          add2(a0, a1, a0, a1, e[u], e[u + 1]);
          add2(a0, a1, a0, a1, e[u + 2], e[u + 3]);
        }
        fp4_p_group(e, max16(e), rho_tab, w);
      } else {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float e[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int u = half * 16 + q4 * 4 + v;
            e[v] = ch * 32 + u < limit ? ex2(fmaf(__uint_as_float(t[u]), cgc, bias)) : 0.f;
          }
          add2(a0, a1, a0, a1, e[0], e[1]);
          add2(a0, a1, a0, a1, e[2], e[3]);
          if constexpr (PV16) {
            w[2 * q4] = pack_p2<true>(e[0], e[1]);
            w[2 * q4 + 1] = pack_p2<true>(e[2], e[3]);
          } else {
            w[q4] = pack_p2<false>(e[0], e[1]) | (pack_p2<false>(e[2], e[3]) << 16);
          }
        }
      }
      store_p_group<PV16>(my_p, r, 2 * ch + half, w);
    }
  }
  return a0 + a1;
}

// P~ = fmt(2^(S * c_g + bias)) of every key of a fully visible tile whose scores sr are in
// registers, written to the row's P buffer; the unquantised values are summed into gsum (four
// independent accumulator pairs).
template <int PV, int DP>
__device__ __forceinline__ void tile_exp_regs(const uint32_t (&sr)[4][32], const float (&cg)[8],
                                              float bias, uint8_t* my_p, int r,
                                              const float* rho_tab, float (&gsum)[8],
                                              const float (&gm)[8]) {
  constexpr bool PV16 = PV != 0, FP4 = PV == 2;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float a0 = 0.f, a1 = 0.f;
    uint32_t w[PV16 ? 8 : 4];
    float eg[FP4 ? 16 : 1];  // FP4: the group's values, quantised once all are known
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int c = g * 16 + q4 * 4;
      float x0, x1, x2, x3;
      fma2(x0, x1, __uint_as_float(sr[c >> 5][c & 31]), __uint_as_float(sr[c >> 5][(c & 31) + 1]),
           cg[g], cg[g], bias, bias);
      fma2(x2, x3, __uint_as_float(sr[c >> 5][(c & 31) + 2]), __uint_as_float(sr[c >> 5][(c & 31) + 3]),
           cg[g], cg[g], bias, bias);
      const float e0 = ex2(x0), e1 = ex2(x1), e2 = ex2(x2), e3 = ex2(x3);
      add2(a0, a1, a0, a1, e0, e1);
      add2(a0, a1, a0, a1, e2, e3);
      if constexpr (FP4) {
        eg[4 * q4] = e0; eg[4 * q4 + 1] = e1; eg[4 * q4 + 2] = e2; eg[4 * q4 + 3] = e3;
      } else if constexpr (PV16) {
        w[2 * q4] = pack_p2<true>(e0, e1);
        w[2 * q4 + 1] = pack_p2<true>(e2, e3);
      } else if constexpr (DP == 64) {
        w[q4] = pack_e4m3x4(e0, e1, e2, e3);
      } else {
        // (the four-value pack measured slower at head_dim 128: c2 0.1206 vs 0.1175 ms)
        w[q4] = pack_p2<false>(e0, e1) | (pack_p2<false>(e2, e3) << 16);
      }
    }
    if constexpr (FP4) {
      // at head_dim 64 the group's largest value is the exponential of its largest score
      // (c_g >= 0, and the fma and the exponential are monotone), one ex2 instead of a max
      // over 16 values; at 128 the maxima come per 32 keys and the 16 values are compared
      fp4_p_group(eg, DP == 64 ? ex2(fmaf(gm[g], cg[g], bias)) : max16(eg), rho_tab, w);
    }
    if constexpr (!PV16 && DP == 64) {
      // (the same swizzled 16-byte unit as store_p_group, addressed in the shared window:
      // measured faster at head_dim 64)
      const uint32_t a = smem_u32(my_p) + static_cast<uint32_t>((g ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                   "r"(w[3]) : "memory");
    } else {
      store_p_group<PV16>(my_p, r, g, w);
    }
    add2(gsum[2 * (g & 3)], gsum[2 * (g & 3) + 1], gsum[2 * (g & 3)], gsum[2 * (g & 3) + 1], a0, a1);
  }
}

// 16 consecutive 32-bit TMEM columns into r[OFF .. OFF + 16) (thread t: lane (lane field of
// taddr) + t), and their maximum as fp32 into m: the reducing form of the load. Both are valid
// only after a tcgen05.wait::ld (tmem_wait_ld for r, tmem_wait_ld_max for m).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_max4(float (&m)[4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+f"(m[0]), "+f"(m[1]), "+f"(m[2]), "+f"(m[3]) : : "memory");
}
template <int OFF>
__device__ __forceinline__ void tmem_ld16_max(uint32_t taddr, uint32_t (&r)[32], float& m) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, %16, [%17];"
      : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]),
        "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]),
        "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]),
        "=r"(r[OFF + 14]), "=r"(r[OFF + 15]), "=f"(m)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_max(float (&m)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(m[0]), "+f"(m[1]), "+f"(m[2]), "+f"(m[3]), "+f"(m[4]), "+f"(m[5]), "+f"(m[6]),
                 "+f"(m[7])
               :
               : "memory");
}

// Max over a fully visible tile of S * c_g, the scores loaded into registers sr (c_g >= 0
// keeps the order). The largest raw integer score of each K scale group's columns comes with
// their load (the reducing form of tcgen05.ld): per 32 columns at head_dim 128 with 64-key K
// groups, per 16 columns otherwise (the 16-column form at head_dim 128 with 64-key groups
// measured slower than the 32-column one).
template <int DP>
__device__ __forceinline__ float tile_max_regs(uint32_t tS, uint32_t (&sr)[4][32], const float (&cg)[8],
                                              int lgk, float (&gm)[8]) {
  if (DP == 128 && lgk == 6) {
    float cm[4];
    tmem_ld32_max(tS + 0, sr[0], cm[0]);
    tmem_ld32_max(tS + 32, sr[1], cm[1]);
    tmem_ld32_max(tS + 64, sr[2], cm[2]);
    tmem_ld32_max(tS + 96, sr[3], cm[3]);
    tmem_wait_ld(sr[0]);
    tmem_wait_ld(sr[1]);
    tmem_wait_ld(sr[2]);
    tmem_wait_ld(sr[3]);
    tmem_wait_ld_max4(cm);
    return fmaxf(fmaxf(cm[0] * cg[0], cm[1] * cg[2]), fmaxf(cm[2] * cg[4], cm[3] * cg[6]));
  }
  {
    tmem_ld16_max<0>(tS + 0, sr[0], gm[0]);
    tmem_ld16_max<16>(tS + 16, sr[0], gm[1]);
    tmem_ld16_max<0>(tS + 32, sr[1], gm[2]);
    tmem_ld16_max<16>(tS + 48, sr[1], gm[3]);
    tmem_ld16_max<0>(tS + 64, sr[2], gm[4]);
    tmem_ld16_max<16>(tS + 80, sr[2], gm[5]);
    tmem_ld16_max<0>(tS + 96, sr[3], gm[6]);
    tmem_ld16_max<16>(tS + 112, sr[3], gm[7]);
    tmem_wait_ld(sr[0]);
    tmem_wait_ld(sr[1]);
    tmem_wait_ld(sr[2]);
    tmem_wait_ld(sr[3]);
    tmem_wait_ld_max(gm);
    float tile_max = __int_as_float(0xff800000);
#pragma unroll
    for (int g = 0; g < 8; ++g) tile_max = fmaxf(tile_max, gm[g] * cg[g]);
    return tile_max;
  }
}

// Records clock64() for (role, tile, event) when tracing is on and this is CTA (0,0,0). Only
// the test instantiation of the kernel (ON = true: pipeline trace and integer-score dump)
// contains the records: a runtime check at every trace point split the softmax loop into basic
// blocks the compiler could not schedule across (measured: 6% of the attention time at
// head_dim 64, 9% at 128).
template <bool ON>
__device__ __forceinline__ void trace(const Problem& p, bool on, int role, int tile, int ev) {
  if constexpr (ON) {
    if (on && tile < kTraceTiles)
      p.dbg_trace[(role * kTraceTiles + tile) * kTraceEvents + ev] = clock64();
  }
}

template <int DP, int PV, bool TRACE>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const Problem p) {
  constexpr bool PV16 = PV != 0;  // P·V on kind::f16 (fp16 P and V^T)
  constexpr bool FP4 = PV == 2;
  using C = AttnCfg<DP, PV16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sP = sm + C::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::kKStages;
  uint64_t* v_full = k_empty + C::kKStages;
  uint64_t* v_empty = v_full + C::kVStages;
  uint64_t* s_full = v_empty + C::kVStages;  // [kSBufs]
  uint64_t* p_full = s_full + C::kSBufs;     // [2]
  uint64_t* o_full = p_full + 2;             // [2]
  uint64_t* o_ready = o_full + 2;            // [2]
  uint64_t* drain = o_ready + 2;             // [2]
  uint64_t* s_free = drain + 2;              // [2] (one S buffer per tile: S read into registers)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  float* rho_tab = reinterpret_cast<float*>(sm + C::kOffRho);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tr = TRACE && p.dbg_trace != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;

  // ---- work item: (query head, 256-row pair, sequence); heaviest pairs first when causal
  // pairs fastest when the host asks for it (non-causal problems whose K / V exceed L2:
  // consecutive CTAs then share one head's K / V there); otherwise heads fastest, heaviest
  // pairs first when causal
  const int lin = (int)blockIdx.x + (int)blockIdx.y * (int)gridDim.x;
  const int h = p.pair_major ? lin / (int)gridDim.y : (int)blockIdx.x;
  const int b = p.varlen ? p.seqinfo[kSiOrder * p.batch + blockIdx.z] : blockIdx.z;
  const Seq s = get_seq(p, b);
  const int npairs_seq = (s.len_q + 2 * kTileRows - 1) / (2 * kTileRows);
  const int pair = p.pair_major ? lin % (int)gridDim.y
                                : (p.is_causal ? (int)gridDim.y - 1 - (int)blockIdx.y : (int)blockIdx.y);
  if (pair >= npairs_seq || s.len_k <= 0) return;  // uniform across the CTA
  const int q_start = pair * 2 * kTileRows;
  const int rows_a = min(kTileRows, s.len_q - q_start);
  const int rows_b = max(0, min(kTileRows, s.len_q - q_start - kTileRows));
  const bool has_b = rows_b > 0;
  const int hk = h / (p.hq / p.hkv);
  const int64_t plane_q = plane_of(p, b, h, p.hq);
  const int64_t plane_kv = plane_of(p, b, hk, p.hkv);
  int kv_end = s.len_k;
  if (p.is_causal) kv_end = min(kv_end, q_start + (has_b ? kTileRows + rows_b : rows_a));
  const int n_tiles = (kv_end + kTileKeys - 1) / kTileKeys;

  // ---- set-up: barriers, tensor memory
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // shared K / V stages are released by each query tile's MMA issuer
    const int k_rel = has_b ? 2 : 1;
    for (int i = 0; i < C::kKStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], k_rel); }
    for (int i = 0; i < C::kVStages; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], k_rel); }
    for (int i = 0; i < C::kSBufs; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_ready[i], 128);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(&s_free[0], 128);
    mbar_init(&s_free[1], 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (FP4 && threadIdx.x < 128) {
    // fl32(6 / s) for the non-negative E4M3 codes (0 for s = 0 and for the NaN code)
    const float sv = __low2float(e4m3x2_to_half2(threadIdx.x * 0x101u));
    rho_tab[threadIdx.x] = (sv > 0.f && threadIdx.x != 0x7f) ? __fdiv_rn(6.0f, sv) : 0.f;
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the quantised operands and scales come from the previous kernel in the stream
  pdl_wait();

  if (warp >= 8) {
   regs_dec<kRegsControl>();
   if (warp == 8) {
    // =========================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int qrow = s.row0_q + q_start;
      mbar_arrive_expect_tx(q_full, (has_b ? 2 : 1) * C::kQTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sQ + c * kTileRows * 128, &tmQ, q_full, c * 64, qrow, (int)plane_q);
        if (has_b)
          tma_load_3d(sQ + C::kQTileBytes + c * kTileRows * 128, &tmQ, q_full, c * 64,
                      qrow + kTileRows, (int)plane_q);
      }
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      if (p.dbg_stall) {
        // test hook: no K/V tile ever arrives, so every consumer wait runs into its bound
        volatile int never = 0;
        mbar_wait(q_full, 0, &never);
      }
      for (int j = 0; j < n_tiles && ok && !p.dbg_stall; ++j) {
        const int krow = s.row0_k + j * kTileKeys;
        const int st = j % C::kKStages;
        if (j >= C::kKStages) ok = mbar_wait(&k_empty[st], ((j / C::kKStages) - 1) & 1, abort_flag);
        if (!ok) break;
        trace<TRACE>(p, tr, 3, j, 0);
        mbar_arrive_expect_tx(&k_full[st], C::kKTileBytes + (C::kKVShared ? C::kVTileBytes : 0));
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK + st * C::kKTileBytes + c * kTileKeys * 128, &tmK, &k_full[st], c * 64,
                      krow, (int)plane_kv);
        ++issued_k;
        const int sv = j % C::kVStages;
        uint64_t* const vbar = C::kKVShared ? &k_full[st] : &v_full[sv];
        if constexpr (!C::kKVShared) {
          if (j >= C::kVStages) ok = mbar_wait(&v_empty[sv], ((j / C::kVStages) - 1) & 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[sv], C::kVTileBytes);
        }
        trace<TRACE>(p, tr, 3, j, 1);
        if constexpr (PV16) {
          // fp16 V^T: two 64-key chunks of DP rows x 128 bytes
          for (int c = 0; c < 2; ++c)
            tma_load_3d(sV + sv * C::kVTileBytes + c * DP * 128, &tmV, vbar, krow + c * 64, 0,
                        (int)plane_kv);
        } else {
          tma_load_3d(sV + sv * C::kVTileBytes, &tmV, vbar, krow, 0, (int)plane_kv);
        }
        ++issued_v;
      }
      if (!ok) {
        // let the copies already in flight land before the CTA's shared memory goes away
        volatile int never = 0;
        mbar_wait(q_full, 0, &never);
        for (int j = max(0, issued_k - C::kKStages); j < issued_k; ++j)
          mbar_wait(&k_full[j % C::kKStages], (j / C::kKStages) & 1, &never);
        if (!C::kKVShared)
          for (int j = max(0, issued_v - C::kVStages); j < issued_v; ++j)
            mbar_wait(&v_full[j % C::kVStages], (j / C::kVStages) & 1, &never);
        record_error(p.err, kDevTimeout);
      }
    }
   } else if (warp == 9 || (warp == 10 && has_b)) {
    // =========================================================== MMA issuer
    // The whole warp runs the issue loop converged and one elected lane issues each MMA and
    // commit (warp-uniform operands). Each query tile has its own issuer; a stage of K / V is
    // released by one commit from each issuer that read it.
    {
      const bool tr_mma = tr && lane == 0;
      const int nx = has_b ? 2 : 1;
      const int me = warp - 9;  // this issuer's query tile
      // descriptor bases; a K step inside a 128-byte row adds its byte offset / 16 to the
      // start-address field (no carry: shared-memory addresses stay below 2^18)
      const uint64_t dq = sdesc_sw128(smem_u32(sQ));
      const uint64_t dk = sdesc_sw128(smem_u32(sK));
      const uint64_t dp = sdesc_sw128(smem_u32(sP));
      const uint64_t dv = sdesc_sw128(smem_u32(sV));
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      // S of query tile x into S buffer sb from K stage st
      auto issue_qk = [&](int x, int sb, int st) {
        const uint32_t d_s = tmem + static_cast<uint32_t>(sb) * 128u;
        const uint64_t qx = dq + static_cast<uint64_t>((x * C::kQTileBytes) >> 4);
        const uint64_t kst = dk + static_cast<uint64_t>((st * C::kKTileBytes) >> 4);
        // K = head_dim in steps of 16 (32 bytes) inside 64-channel chunks of 128-byte rows; at
        // head_dim 64 the four MMAs from one elected block (measured faster there, not at 128)
        if constexpr (DP == 64) {
          mma4_warp<false>(d_s, qx, qx + 2, qx + 4, qx + 6, kst, kst + 2, kst + 4, kst + 6, idesc_qk(), 0u);
        } else {
#pragma unroll
          for (int k = 0; k < DP / 16; ++k) {
            const uint32_t off = ((k >> 2) * (kTileRows * 128) + (k & 3) * 32) >> 4;
            mma_f16_ss_warp(d_s, qx + off, kst + off, idesc_qk(), k > 0);
          }
        }
        mma_commit_warp(&s_full[sb]);
      };
      auto issue_pv = [&](int x, int sv, int buf, bool first) {
        const uint32_t d_o = tmem + C::kTmemO + static_cast<uint32_t>(x * DP);
        const uint64_t px =
            dp + static_cast<uint64_t>(((x * C::kPBufs + buf) * C::kPTileBytes) >> 4);
        const uint64_t vst = dv + static_cast<uint64_t>((sv * C::kVTileBytes) >> 4);
        if constexpr (PV16) {
          // K = 128 keys in steps of 16 (32 bytes) inside 64-key chunks
          if constexpr (DP == 64) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint32_t op = (c * (kTileRows * 128)) >> 4;
              const uint32_t ov = (c * (DP * 128)) >> 4;
              mma4_warp<false>(d_o, px + op, px + op + 2, px + op + 4, px + op + 6, vst + ov, vst + ov + 2,
                               vst + ov + 4, vst + ov + 6, idesc_pv<DP>(), (!first || c > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kTileKeys / 16; ++k) {
              const uint32_t op = ((k >> 2) * (kTileRows * 128) + (k & 3) * 32) >> 4;
              const uint32_t ov = ((k >> 2) * (DP * 128) + (k & 3) * 32) >> 4;
              mma_f16_ss_warp(d_o, px + op, vst + ov, idesc_pv<DP>(), (!first || k > 0) ? 1u : 0u);
            }
          }
        } else {
          if constexpr (DP == 64) {
            mma4_warp<true>(d_o, px, px + 2, px + 4, px + 6, vst, vst + 2, vst + 4, vst + 6, idesc_pv<DP>(),
                            first ? 0u : 1u);
          } else {
#pragma unroll
            for (int k = 0; k < kTileKeys / 32; ++k)
              mma_f8_ss_warp(d_o, px + 2 * k, vst + 2 * k, idesc_pv<DP>(), (!first || k > 0) ? 1u : 0u);
          }
        }
        mma_commit_warp(&o_full[x]);
      };
      bool ok = wait_all(q_full, 0);
      if constexpr (C::kSBufs == 3) {
        // Items n = j * nx + x in order. Once the softmax of item n has published P (its S
        // buffer is free and, for j > 0, its O rows are rescaled), P_j(x) V_j is issued and
        // the scores of item n + 3 go into that buffer (the other query tile's next tile when
        // both exist, which its softmax needs only after its current tile).
        const int n_items = n_tiles * nx;
        const int lnx = nx - 1;  // log2(nx): items n = j * nx + x
        // QK^T of item n into S buffer n % 3 (after this issuer's own wait for K_kj: the
        // other issuer's wait orders nothing for this thread)
        auto qk_item = [&](int n) {
          const int kj = n >> lnx, xx = n & lnx, st = kj % C::kKStages;
          if (!wait_all(&k_full[st], (kj / C::kKStages) & 1)) return false;
          tc_fence_after();
          issue_qk(xx, n % 3, st);
          return true;
        };
        if (me == 0) {
          for (int n = 0; n < 3 && n < n_items && ok; ++n) ok = qk_item(n);
        } else {
          // the stages of tiles 0 and 1 are first read by this issuer's P.V
          for (int kj = 0; kj < 2 && kj < n_tiles && ok; ++kj) {
            ok = wait_all(&k_full[kj], 0);
            if (ok) tc_fence_after();
          }
        }
        // each issuer walks its own query tile's items; the scores of item n + 3 (the other
        // tile's, when both exist) are issued by the issuer of item n
        for (int n = me; n < n_items && ok; n += nx) {
          const int j = n >> lnx, x = me, sv = j % C::kVStages;
          ok = wait_all(&p_full[x], j & 1);
          if (!ok) break;
          trace<TRACE>(p, tr_mma, 2, j, 4 * x + 0);
          tc_fence_after();
          // P_j(x) V_j first (the softmax waits for it before publishing its next P, or with
          // one P buffer before its next exponentials), then the scores three items ahead
          // (V_j arrived with K_j, which this issuer waited for at an earlier item)
          trace<TRACE>(p, tr_mma, 2, j, 4 * x + 1);
          issue_pv(x, sv, j % C::kPBufs, j == 0);
          mma_commit_warp(&k_empty[sv]);  // this issuer's last use of K_j and V_j
          trace<TRACE>(p, tr_mma, 2, j, 4 * x + 2);
          if (n + 3 < n_items) ok = qk_item(n + 3);
          trace<TRACE>(p, tr_mma, 2, j, 4 * x + 3);
        }
      } else {
      if (ok) ok = wait_all(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_qk(me, me, 0);
        mma_commit_warp(&k_empty[0]);
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int sv = j % C::kVStages;
        const int nst = (j + 1) % C::kKStages;
        const int x = me;
        if (j + 1 < n_tiles) {
          // S_j(x) is in the softmax's registers: the tile's next scores can start
          ok = wait_all(&s_free[x], j & 1);
          if (!ok) break;
          trace<TRACE>(p, tr_mma, 2, j, 4 * x + 0);
          ok = wait_all(&k_full[nst], ((j + 1) / C::kKStages) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_qk(x, x, nst);
          mma_commit_warp(&k_empty[nst]);
        }
        trace<TRACE>(p, tr_mma, 2, j, 4 * x + 1);
        // P_j(x) written and O(x) rescaled for the new running max: accumulate P_j(x) V_j
        ok = wait_all(&o_ready[x], j & 1);
        if (!ok) break;
        trace<TRACE>(p, tr_mma, 2, j, 4 * x + 2);
        ok = wait_all(&v_full[sv], (j / C::kVStages) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_pv(x, sv, j % C::kPBufs, j == 0);
        mma_commit_warp(&v_empty[sv]);
        trace<TRACE>(p, tr_mma, 2, j, 4 * x + 3);
      }
      }
      // every MMA must have finished before tensor memory is released
      mma_commit_warp(&drain[me]);
      volatile int never = 0;
      mbar_wait(&drain[me], 0, &never);
      __syncwarp();
      if (!ok && lane == 0) record_error(p.err, kDevTimeout);
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // =========================================================== softmax (warps 0-7)
    const int x = warp >> 2;               // tile A or B
    const int r = (warp & 3) * 32 + lane;  // row in tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    constexpr bool kRing = C::kSBufs == 3;  // S buffers in rotation (head_dim 64)
    const int nx = has_b ? 2 : 1;
    const uint32_t tO = tmem + lane_base + C::kTmemO + static_cast<uint32_t>(x * DP);
    // this query tile's S buffer (head_dim 128; at 64 the buffer rotates per tile)
    uint32_t tS = tmem + lane_base + (x == 0 ? 0u : 128u);
    uint8_t* const p_row = sP + x * C::kPBufs * C::kPTileBytes + r * 128;  // + buffer offset
    const int xrows = x == 0 ? rows_a : rows_b;
    const bool active_tile = x == 0 || has_b;
    const int i = q_start + x * kTileRows + r;  // query row within the sequence
    const bool row_valid = active_tile && r < xrows;
    // sigma_P: 448 (the largest E4M3 magnitude) for E4M3 P in every accumulation mode, 1 for
    // fp16 P
    const float log2_sigma = (PV16 && !FP4) ? 0.0f : 8.807354922057604f;  // log2(448)
    const bool trs = tr && (warp & 3) == 0 && lane == 0;
    float sq = 0.f;
    if (row_valid) sq = __ldg(&p.sq[plane_q * p.sq_pp + (s.row0_q + i) / p.gq]);
    // FP4: the carriers are ~6x the mapped values on both sides, so the scores carry 36
    const float row_scale = sq * p.sm_scale * (FP4 ? kLog2e / 36.0f : kLog2e);
    const float* skp = p.sk + plane_kv * p.sk_pp + (s.row0_k >> p.lgk);
    const int lgk = p.lgk;  // log2 of the K scale group (16 or 64 keys)
    float m = __int_as_float(0xff800000);  // running max (log2 units)
    float l = 0.f;                          // running sum of 2^(x - m) * sigma
    bool ok = true;
    // K scales of the 8 sub-groups of 16 keys, loaded one tile ahead of their use
    float skn[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) skn[g] = g * 16 < s.len_k ? __ldg(&skp[(g * 16) >> lgk]) : 0.f;
    // keys this row may see: [0, row_limit) (causal: j <= i; always: j < len_k)
    const int row_limit = p.is_causal ? min(s.len_k, i + 1) : s.len_k;
    // S buffer (item n = j * nx + x mod 3) and its phase parity ((n / 3) mod 2), advanced by nx
    // items per tile
    int s_buf = x, s_par = 0;
    if (active_tile) {
      for (int j = 0; j < n_tiles; ++j) {
        if constexpr (kRing) {
          tS = tmem + lane_base + static_cast<uint32_t>(s_buf) * 128u;
          ok = __all_sync(0xffffffffu, mbar_wait(&s_full[s_buf], s_par, abort_flag));
          s_buf += nx;
          if (s_buf >= 3) {
            s_buf -= 3;
            s_par ^= 1;
          }
        } else {
          ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1, abort_flag));
        }
        if (!ok) break;
        trace<TRACE>(p, trs, x, j, 0);
        tc_fence_after();
        const int kv0 = j * kTileKeys;
        const int limit = row_limit - kv0;  // this row's allowed keys in the tile: [0, limit)
        const bool masked = __any_sync(0xffffffffu, limit < kTileKeys);
        if constexpr (TRACE || DP == 128) {  // (head_dim 128: measured faster with the check)
          if (p.dbg_scores != nullptr)
            dump_scores_row(tS, row_valid, p.dbg_scores + ((int64_t)(b * p.hq + h) * p.nq + i) * p.nk + kv0,
                            min(kTileKeys, s.len_k - kv0));
        }
        // multipliers c_g = s_q * s_k * sm_scale * log2(e) for the 8 sub-groups of 16 keys
        // (a K scale group is 16 or 64 keys, so each sub-group has one scale)
        float cg[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) cg[g] = row_scale * skn[g];
        uint32_t sr[4][32];
        float gmx[8];  // the scores' 16-key group maxima (unmasked tiles)
        float tile_max = __int_as_float(0xff800000);
        float m_new, alpha, bias;
        uint8_t* const my_p = p_row + (j % C::kPBufs) * C::kPTileBytes;
        float gsum[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) gsum[u] = 0.f;
        Mult8 c8;  // the masked paths' copy of c_g
#pragma unroll
        for (int g = 0; g < 8; ++g) c8.v[g] = cg[g];
        // the new running max, the rescale factor and the exponent bias; with one P buffer the
        // buffer is free once P.V of tile j - 1 has completed (with two, P.V of tile j - 2, its
        // previous reader, completed before this row's rescale wait of tile j - 1 below)
        auto new_max = [&]() {
          m_new = fmaxf(m, tile_max);
          const float m_use = m_new == __int_as_float(0xff800000) ? 0.f : m_new;
          alpha = ex2(m - m_use);  // 0 on the first tile (m = -inf)
          bias = log2_sigma - m_use;
          if (C::kPBufs == 1 && j > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&o_full[x], (j - 1) & 1, abort_flag));
            if (ok) tc_fence_after();
          }
        };
        // The unmasked path (every key of the tile visible, causal diagonal and ragged tail
        // excepted) either runs as one branch from the loads to the last P store (head_dim
        // 64) or as two branches joined around the max (head_dim 128): measured, each is the
        // faster arrangement for its head_dim (c4 attention 8.84 vs 8.90 ms; c2 0.1235 vs
        // 0.1278 ms)
        if constexpr (DP == 64) {
          if (__builtin_expect(!masked, 1)) {
            tile_max = tile_max_regs<DP>(tS, sr, cg, lgk, gmx);
            trace<TRACE>(p, trs, x, j, 1);
            trace<TRACE>(p, trs, x, j, 2);
            new_max();
            trace<TRACE>(p, trs, x, j, 4);
            if (ok) tile_exp_regs<PV, DP>(sr, cg, bias, my_p, r, rho_tab, gsum, gmx);
          } else {
            tile_max = masked_tile_max(tS, limit, c8);
            trace<TRACE>(p, trs, x, j, 1);
            trace<TRACE>(p, trs, x, j, 2);
            new_max();
            trace<TRACE>(p, trs, x, j, 4);
            if (ok) gsum[0] = masked_tile_exp<PV>(tS, limit, c8, bias, my_p, r, rho_tab);
          }
          if (!ok) break;
        } else {
          if (__builtin_expect(!masked, 1)) {
            tile_max = tile_max_regs<DP>(tS, sr, cg, lgk, gmx);
            tc_fence_before();
            mbar_arrive(&s_free[x]);
          } else {
            tile_max = masked_tile_max(tS, limit, c8);
          }
          trace<TRACE>(p, trs, x, j, 1);
          trace<TRACE>(p, trs, x, j, 2);
          new_max();
          if (!ok) break;
          trace<TRACE>(p, trs, x, j, 4);
          if (__builtin_expect(!masked, 1)) {
            tile_exp_regs<PV, DP>(sr, cg, bias, my_p, r, rho_tab, gsum, gmx);
          } else {
            gsum[0] = masked_tile_exp<PV>(tS, limit, c8, bias, my_p, r, rho_tab);
            tc_fence_before();
            mbar_arrive(&s_free[x]);
          }
        }
        const float rs = ((gsum[0] + gsum[1]) + (gsum[2] + gsum[3])) + ((gsum[4] + gsum[5]) + (gsum[6] + gsum[7]));
        // next tile's K scales (used one tile from now): two loads when a K scale group is
        // 64 keys, eight when it is 16
        if (lgk == 6) {
          const int kg = kv0 + kTileKeys;
          const float s0 = kg < s.len_k ? __ldg(&skp[kg >> 6]) : 0.f;
          const float s1 = kg + 64 < s.len_k ? __ldg(&skp[(kg >> 6) + 1]) : 0.f;
#pragma unroll
          for (int g = 0; g < 8; ++g) skn[g] = g < 4 ? s0 : s1;
        } else {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const int kg = kv0 + kTileKeys + g * 16;
            skn[g] = kg < s.len_k ? __ldg(&skp[kg >> lgk]) : 0.f;
          }
        }
        trace<TRACE>(p, trs, x, j, 3);
        l = l * alpha + rs;
        m = m_new;
        trace<TRACE>(p, trs, x, j, 5);
        // rescale this warp's O rows for the grown max: O holds the sum up to tile j - 1 once
        // P.V of tile j - 1 is complete. P_j(x) V_j is issued only after the rescale: with one
        // S buffer per tile (head_dim 128) o_ready carries P_j and the rescaled O together; with
        // the S buffers in rotation P_j(x) is published after it, and the wait for P.V of tile
        // j - 1 also keeps p_full at most one phase ahead of the MMA issuer.
        if (C::kPBufs > 1 && j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&o_full[x], (j - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha < 1.0f)) {
#pragma unroll
          for (int c2 = 0; c2 < DP / 64; ++c2) {
          uint32_t o[2][32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) tmem_ld32(tO + (c2 * 2 + cc) * 32, o[cc]);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) tmem_wait_ld(o[cc]);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int u = 0; u < 32; u += 2) {
              float a0, a1;
              mul2(a0, a1, __uint_as_float(o[cc][u]), __uint_as_float(o[cc][u + 1]), alpha, alpha);
              o[cc][u] = __float_as_uint(a0);
              o[cc][u + 1] = __float_as_uint(a1);
            }
            tmem_st32(tO + (c2 * 2 + cc) * 32, o[cc]);
          }
          }
          tmem_wait_st();
        }
        if constexpr (kRing) {
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&p_full[x]);
          trace<TRACE>(p, trs, x, j, 5);
        } else {
          // P_j(x) and the rescaled O together
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&o_ready[x]);
        }
        trace<TRACE>(p, trs, x, j, 6);
      }
      // ---- epilogue: out = acc . s_v / l + v_mean, then the LSE. The output address, the LSE
      // term and the first chunk's V scales / means are fetched while P.V of the last tile
      // completes, and each 32-channel chunk's scales are requested before the previous
      // chunk's values are stored. The chunk loop stays rolled: it runs once per CTA, from a
      // cold instruction cache. Rows of 16-byte chunks (head_dim % 8 == 0) are stored 16
      // bytes at a time; with head_dim 64 each thread first puts its row into this tile's P
      // buffers (free once the last P.V is done), XOR-swizzled by chunk so that neither side
      // conflicts on banks, and each warp then writes its 32 rows out whole, four rows per
      // store instruction (measured: faster than direct row stores for head_dim 64, slower
      // for 128).
      const float* vsc = p.vscale + ((int64_t)b * p.hkv + hk) * p.d;
      const float* vmn = p.vmean + ((int64_t)b * p.hkv + hk) * p.d;
      uint16_t* const dst = static_cast<uint16_t*>(p.o) + (int64_t)b * p.o_sb +
                            (int64_t)(s.tok0_q + i) * p.o_sn + (int64_t)h * p.o_sh;
      constexpr bool kStageOut = DP == 64;
      constexpr int kSwz = DP / 8 - 1;  // 16-byte chunks of a staged row, minus one
      uint8_t* const stage = sP + x * C::kPBufs * C::kPTileBytes;  // [128 rows][DP * 2 bytes]
      static_assert(kTileRows * DP * 2 <= C::kPBufs * C::kPTileBytes, "output staging fits in P");
      const bool vec = p.vec16 != 0;  // head_dim % 8 == 0, 16-byte aligned output rows
      float qk_term = 0.f;
      if (p.return_lse && p.smooth_k && row_valid) qk_term = p.qkc[plane_q * p.q_rows + s.row0_q + i];
      float4 cs[8], cm[8];  // V scales / means of the current chunk's 32 channels
      if (vec) load_chunk_scales(vsc, vmn, 0, p.d, cs, cm);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[x], (n_tiles - 1) & 1, abort_flag));
      if (ok) {
        tc_fence_after();
        // FP4: O = acc . s_v / (36 l) (both P·V carriers are ~6x their mapped values)
        const float inv_l = 1.0f / (FP4 ? 36.0f * l : l);
#pragma unroll 1
        for (int cc = 0; cc < DP / 32 && cc * 32 < p.d; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          float4 ns[8], nm[8];
          const bool more = vec && cc + 1 < DP / 32 && (cc + 1) * 32 < p.d;
          if (more) load_chunk_scales(vsc, vmn, (cc + 1) * 32, p.d, ns, nm);
          tmem_wait_ld(o);
          if (row_valid) {
            if (vec) {
              // whole 8-channel groups (head_dim % 8 == 0), one 16-byte store each
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (cc * 32 + q * 8 < p.d) {
                  const float4 s0 = cs[2 * q], s1 = cs[2 * q + 1], m0 = cm[2 * q], m1 = cm[2 * q + 1];
                  const float* ov = reinterpret_cast<const float*>(o) + q * 8;
                  uint4 w;
                  w.x = pack_out2(fmaf(ov[0] * s0.x, inv_l, m0.x), fmaf(ov[1] * s0.y, inv_l, m0.y), p.dtype);
                  w.y = pack_out2(fmaf(ov[2] * s0.z, inv_l, m0.z), fmaf(ov[3] * s0.w, inv_l, m0.w), p.dtype);
                  w.z = pack_out2(fmaf(ov[4] * s1.x, inv_l, m1.x), fmaf(ov[5] * s1.y, inv_l, m1.y), p.dtype);
                  w.w = pack_out2(fmaf(ov[6] * s1.z, inv_l, m1.z), fmaf(ov[7] * s1.w, inv_l, m1.w), p.dtype);
                  const int c16 = cc * 4 + q;
                  if constexpr (kStageOut)
                    *reinterpret_cast<uint4*>(stage + r * (DP * 2) + ((c16 ^ (r & kSwz)) << 4)) = w;
                  else
                    *reinterpret_cast<uint4*>(dst + c16 * 8) = w;
                }
              }
            } else {
              // element stores: head_dim not a multiple of 8, or unaligned output rows
#pragma unroll 1
              for (int u = 0; u < 32 && cc * 32 + u < p.d; ++u) {
                const int c = cc * 32 + u;
                const float v = fmaf(__uint_as_float(pick32(o, u)) * __ldg(&vsc[c]), inv_l, __ldg(&vmn[c]));
                dst[c] = static_cast<uint16_t>(pack_out2(v, 0.f, p.dtype) & 0xffffu);
              }
            }
          }
          if (more) {
#pragma unroll
            for (int u = 0; u < 8; ++u) { cs[u] = ns[u]; cm[u] = nm[u]; }
          }
        }
        if (kStageOut && vec) {
          // this warp's 32 staged rows to global memory, whole rows per lane group
          __syncwarp();
          const int nch = p.d >> 3;                        // 16-byte chunks of an output row
          const int lg = (nch & (nch - 1)) == 0 ? __ffs(nch) - 1 : -1;
          const int r0 = (warp & 3) * 32;
          const int64_t row_stride = p.o_sn;
          uint16_t* const dst0 = dst - (int64_t)lane * row_stride;  // row r0 of this warp
#pragma unroll 1
          for (int t = lane; t < 32 * nch; t += 32) {
            const int rr = lg >= 0 ? t >> lg : t / nch;
            const int c16 = t - rr * nch;
            const int rw = r0 + rr;
            if (rw < xrows) {
              const uint4 v = *reinterpret_cast<const uint4*>(stage + rw * (DP * 2) + ((c16 ^ (rw & kSwz)) << 4));
              *reinterpret_cast<uint4*>(dst0 + (int64_t)rr * row_stride + c16 * 8) = v;
            }
          }
        }
        if (p.return_lse && row_valid) {
          const float lse = (m + __log2f(l) - log2_sigma) * 0.6931471805599453f + p.sm_scale * qk_term;
          const int64_t li = p.varlen ? (int64_t)h * p.lse_plane + s.tok0_q + i
                                      : ((int64_t)b * p.hq + h) * p.nq + i;
          p.lse[li] = lse;
        }
        trace<TRACE>(p, trs, x, n_tiles - 1, 7);
      }
      if (!ok) record_error(p.err, kDevTimeout);
    }
  }

  // ---- teardown: every role is done with tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
template <int DP, int PV, bool TRACE = false>
static cudaError_t launch_attn_t(const Problem& p, const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
  constexpr int smem = AttnCfg<DP, PV != 0>::kSmem;
  static std::atomic<int> limits[64];
  cudaError_t e = raise_smem_limit(attn_kernel<DP, PV, TRACE>, smem, limits);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<DP, PV, TRACE>, grid, dim3(kAttnThreads), smem, stream, maps[0],
                    maps[1], maps[2], p);
}

cudaError_t launch_attention(const Problem& p, const CUtensorMap* maps, int grid_pairs,
                             cudaStream_t stream) {
  const dim3 grid(p.hq, grid_pairs, p.batch);
  // the test instantiation (pipeline trace, integer-score dump) exists for the E4M3 P·V kernel
  if ((p.dbg_trace != nullptr || p.dbg_scores != nullptr) && !p.pv16)
    return p.dp == 64 ? launch_attn_t<64, 0, true>(p, maps, grid, stream)
                      : launch_attn_t<128, 0, true>(p, maps, grid, stream);
  if (p.fp4) return p.dp == 64 ? launch_attn_t<64, 2>(p, maps, grid, stream)
                               : launch_attn_t<128, 2>(p, maps, grid, stream);
  if (p.pv16) return p.dp == 64 ? launch_attn_t<64, 1>(p, maps, grid, stream)
                                : launch_attn_t<128, 1>(p, maps, grid, stream);
  return p.dp == 64 ? launch_attn_t<64, 0>(p, maps, grid, stream)
                    : launch_attn_t<128, 0>(p, maps, grid, stream);
}

}  // namespace sage
