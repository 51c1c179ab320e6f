// Short-sequence path: the whole forward (K/V statistics, Q/K/V quantisation, attention) in one
// launch, for problems whose keys fit in shared memory (pnsm.cn "SageAttention on AMD 9070 XT
// without the HIP SDK" §10: below about 1K tokens the quantised kernel gains little, because
// fixed costs dominate; pwwt.cn guide §5.1 presents the method as a drop-in for every
// attention call, short ones included).
//
// The main pipeline spends four kernel launches and a clear on every call; for a 256-token
// problem those fixed costs are the whole call. Here one CTA owns 128 query rows of one
// (batch, query head) and does everything itself:
//   0. its KV head's K and V rows into shared memory (cp.async, all in flight at once) and its
//      Q rows into registers;
//   1. the smoothing means of K and V (exact fixed-point sums) and V's per-channel scale,
//      exactly as the statistics / finalisation kernels compute them;
//   2. INT8 codes of K (per key group) and E4M3 codes of V into shared memory, and INT8
//      codes of its Q rows, with the quantisation kernel's arithmetic (bit-identical codes);
//   3. per warp of 16 query rows: QK^T on mma.sync m16n8k16 with the INT8 codes held as fp16
//      (every product and partial sum is an integer below 2^24, exact in the fp32
//      accumulator; the s8 form of the instruction measured 12x slower per instruction on
//      this GPU: 65.6 cycles per m16n8k32 against 5.5 for e4m3), the online softmax over
//      128-key tiles (the same form as the main kernel: P~ against the running maximum of the
//      tiles seen so far), P~ = e4m3(2^(x - m) 448) and P~ V on mma.sync m16n8k32 e4m3 with
//      fp32 accumulation, then O = acc s_v / l + v_mean and the LSE.
// The CTAs of one KV head each requantise its K and V (a few hundred KB from L2 at this size);
// one of them also writes the codes, scales and means into the workspace in the main
// pipeline's layout, so the quantised state can be read back the same way.
// Measured (GB300, 256^2 at head_dim 64): 28.4 us per direct call against 36.8 for the main
// pipeline's four launches, so it is the default there; replayed from a CUDA graph the four
// launches are faster (21.7 us against 26.7), and at head_dim 128 they are faster either way,
// so captured calls and head_dim 128 take the main pipeline. A clock64 trace of one CTA
// (256 keys, ~46,000 cycles) spends about a third in the attention loop and the rest in the
// serial statistics and quantisation passes, each latency-bound from a cold instruction cache.
#include "launch.h"
#include "problem.cuh"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

constexpr int kSRows = 128;     // query rows per CTA: 8 warps x 16 rows
constexpr int kSThreads = 256;
constexpr int kSTile = 128;     // keys per online-softmax tile
constexpr float kSLog2e = 1.4426950408889634f;
constexpr float kSLog2Sigma = 8.807354922057604f;  // log2(448)

__device__ __forceinline__ float ex2s(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D (16x8 fp32) += A (16x32 e4m3, row) * B (32x8 e4m3, col).
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Position of key n in the V^T shared-memory rows. The accumulator fragment of a QK^T tile
// gives lane (g, q) (g = lane / 4, q = lane % 4) the keys 8 t + 2 q + {0, 1} of the four
// 8-key column tiles t of a 32-key chunk; packed as an A fragment of the P.V instruction,
// its k-slots 4 q .. 4 q + 3 then hold keys 2 q, 2 q + 1, 8 + 2 q, 9 + 2 q (tiles 0 and 1) and
// slots 16 + 4 q .. the same keys + 16 (tiles 2 and 3). V rows are stored in that slot order,
// so no value has to move between lanes.
__device__ __forceinline__ int v_slot(int n) {
  const int k = n & 31, t = k >> 3, q = (k >> 1) & 3;
  return (n & ~31) + (t >> 1) * 16 + q * 4 + (t & 1) * 2 + (k & 1);
}

struct ShortSmem {
  int dps, nks, nk_pad;
  uint8_t* rawk;   // [nk_pad][DP] K as loaded (fp16 / bf16), zero beyond the keys and head_dim
  uint8_t* rawv;   // [nk_pad][DP] V likewise
  uint8_t* kcode;  // the raw V space, once V is coded: the K codes as fp16, 16-byte units
                   // XOR-swizzled by (key & 7) so that the MMA fragment loads hit every bank
  uint8_t* vt8;    // [DP][nks]      V^T E4M3 codes, keys in slot order
  __half* q16;     // [128][DP]      Q codes of the CTA's rows (fp16)
  float *kmean, *vmean, *vscale, *vrcp;   // [DP]
  long long *red_k, *red_v;               // [8 warps][DP] statistics partials, in the V^T / Q
  float *red_mn, *red_mx;                 // code space (free until the codes are written)
  unsigned *kgmax, *qgmax;                // [nk_pad / 16], [128] group maxima of |x| (float bits)
  float *gscale, *grcp;                   // [nk_pad / 16] K group scale, reciprocal
  float *qscale, *qrcp, *qkt;             // [128] per Q row: its group's scale, reciprocal, LSE term
};

// Byte offsets of the shared-memory arrays for nk_pad keys; returns the total size.
struct ShortOffsets {
  size_t rawk, rawv, vt8, q16, kmean, vmean, vscale, vrcp, gscale, grcp,
      qscale, qrcp, qkt, kgmax, qgmax, total;
};
__host__ __device__ inline ShortOffsets short_offsets(int dp, int nk_pad) {
  ShortOffsets f;
  const size_t nks = nk_pad + 16;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += (bytes + 15) / 16 * 16; return at; };
  f.rawk = take((size_t)nk_pad * dp * 2);
  f.rawv = take((size_t)nk_pad * dp * 2);
  f.vt8 = take((size_t)dp * nks);
  f.q16 = take((size_t)kSRows * dp * 2);
  f.kmean = take(4 * dp);
  f.vmean = take(4 * dp);
  f.vscale = take(4 * dp);
  f.vrcp = take(4 * dp);

  f.gscale = take(4 * (nk_pad / 16));
  f.grcp = take(4 * (nk_pad / 16));
  f.qscale = take(4 * kSRows);
  f.qrcp = take(4 * kSRows);
  f.qkt = take(4 * kSRows);
  f.kgmax = take(4 * (nk_pad / 16));
  f.qgmax = take(4 * kSRows);
  f.total = o;
  return f;
}

__device__ inline ShortSmem short_smem(int dp, int nk_pad, uint8_t* base) {
  const ShortOffsets f = short_offsets(dp, nk_pad);
  ShortSmem L;
  L.dps = dp + 16;
  L.nks = nk_pad + 16;
  L.nk_pad = nk_pad;
  L.rawk = base + f.rawk;
  L.rawv = base + f.rawv;
  L.kcode = base + f.rawv;
  L.vt8 = base + f.vt8;
  L.q16 = reinterpret_cast<__half*>(base + f.q16);
  L.kmean = reinterpret_cast<float*>(base + f.kmean);
  L.vmean = reinterpret_cast<float*>(base + f.vmean);
  L.vscale = reinterpret_cast<float*>(base + f.vscale);
  L.vrcp = reinterpret_cast<float*>(base + f.vrcp);
  // the statistics partials take 192 dp bytes of the V^T and Q code space (contiguous, at least
  // dp * (nk_pad + 16 + 256) bytes)
  L.red_k = reinterpret_cast<long long*>(base + f.vt8);
  L.red_v = L.red_k + 8 * dp;
  L.red_mn = reinterpret_cast<float*>(L.red_v + 8 * dp);
  L.red_mx = L.red_mn + 8 * dp;
  L.kgmax = reinterpret_cast<unsigned*>(base + f.kgmax);
  L.qgmax = reinterpret_cast<unsigned*>(base + f.qgmax);
  L.gscale = reinterpret_cast<float*>(base + f.gscale);
  L.grcp = reinterpret_cast<float*>(base + f.grcp);
  L.qscale = reinterpret_cast<float*>(base + f.qscale);
  L.qrcp = reinterpret_cast<float*>(base + f.qrcp);
  L.qkt = reinterpret_cast<float*>(base + f.qkt);
  return L;
}

// rint_even(fl32(x * r)) clamped to [-127, 127], as the quantisation kernel computes it
__device__ __forceinline__ int int8_code(float x, float r) {
  float c = __fsub_rn(__fadd_rn(__fmul_rn(x, r), kRoundMagic), kRoundMagic);
  c = fminf(fmaxf(c, -127.0f), 127.0f);
  return static_cast<int>(c);
}

template <typename T, int DP>
__global__ void __launch_bounds__(kSThreads, 1) short_attn_kernel(const Problem p) {
  constexpr int TPR = DP / 8;            // threads per row (8 channels each)
  constexpr int RG = kSThreads / TPR;    // rows per pass
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int nk = p.nk, nq = p.nq, d = p.d;
  const int nk_pad = (nk + kSTile - 1) / kSTile * kSTile;
  const ShortSmem S = short_smem(DP, nk_pad, smem_raw);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int vec = t % TPR, rg = t / TPR, c0 = vec * 8;
  const int h = blockIdx.y, b = blockIdx.z;
  const int grp = p.hq / p.hkv, hk = h / grp;
  const int r0 = blockIdx.x * kSRows;
  // one CTA per KV head writes the K / V codes, scales and means to the workspace
  const bool kv_writer = blockIdx.x == 0 && h % grp == 0;
  const int64_t plane_q = (int64_t)b * p.hq + h, plane_kv = (int64_t)b * p.hkv + hk;
  const int64_t sidx = plane_kv * d;
  const T* kb = static_cast<const T*>(p.k) + (int64_t)b * p.k_sb + (int64_t)hk * p.k_sh;
  const T* vb = static_cast<const T*>(p.v) + (int64_t)b * p.v_sb + (int64_t)hk * p.v_sh;
  const T* qb = static_cast<const T*>(p.q) + (int64_t)b * p.q_sb + (int64_t)h * p.q_sh;

  // ---- 0. loads: K and V rows into shared memory (cp.async, all in flight at once), this
  // CTA's Q rows into registers; every later pass reads these copies
  constexpr int QPT = kSRows / RG;  // Q rows per thread
  uint4 qraw[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = r0 + rg + RG * u;
    qraw[u] = i < nq ? load8_raw<T>(qb + (int64_t)i * p.q_sn, c0, d, p.vec16) : make_uint4(0, 0, 0, 0);
  }
  const bool full_vec = p.vec16 && c0 + 8 <= d;
  for (int n = rg; n < nk_pad; n += RG) {
    uint8_t* dk = S.rawk + ((size_t)n * DP + c0) * 2;
    uint8_t* dv = S.rawv + ((size_t)n * DP + c0) * 2;
    if (n < nk && full_vec) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dk)),
                   "l"(kb + (int64_t)n * p.k_sn + c0) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dv)),
                   "l"(vb + (int64_t)n * p.v_sn + c0) : "memory");
    } else {
      *reinterpret_cast<uint4*>(dk) = n < nk ? load8_raw<T>(kb + (int64_t)n * p.k_sn, c0, d, p.vec16) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(dv) = n < nk ? load8_raw<T>(vb + (int64_t)n * p.v_sn, c0, d, p.vec16) : make_uint4(0, 0, 0, 0);
    }
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  for (int g = t; g < nk_pad / 16; g += kSThreads) S.kgmax[g] = 0u;
  for (int g = t; g < kSRows; g += kSThreads) S.qgmax[g] = 0u;
  // the status word is cleared by the launch before this one (which may still be finishing):
  // nothing in the workspace is touched before it has
  pdl_wait();
  __syncthreads();
  auto row8 = [&](const uint8_t* raw, int n, float (&x)[8]) {
    unpack8<T>(*reinterpret_cast<const uint4*>(raw + ((size_t)n * DP + c0) * 2), x);
  };

  // ---- 1. statistics: exact fixed-point sums of K and V, V's min / max per channel (the
  // sums as biased 32-bit split words, as the statistics kernel forms them); and the Q group
  // maxima (Q needs no statistics)
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    float x[8], a = 0.f;
    unpack8<T>(qraw[u], x);
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(x[j]));
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (p.gq == 1) {
      if (vec == 0) S.qgmax[rg + RG * u] = __float_as_uint(a);  // one row per group
    } else {
      // Q groups of 32 or 128 rows hold the warp's 32 / TPR consecutive rows
#pragma unroll
      for (int off = TPR; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
      if (lane == 0) atomicMax(&S.qgmax[(rg + RG * u) / p.gq], __float_as_uint(a));
    }
  }
  {
    unsigned kh[8], kl[8], vh[8], vl[8];
    float mn[8], mx[8], amax = 0.f;
    bool exact = true;
    int nrows = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      kh[i] = kl[i] = vh[i] = vl[i] = 0u;
      mn[i] = __int_as_float(0x7f800000);
      mx[i] = __int_as_float(0xff800000);
    }
    // the row loops of the statistics and code passes are unrolled so that independent rows'
    // shared-memory loads and reductions overlap
#pragma unroll 4
    for (int n = rg; n < nk; n += RG) {
      float xk[8], xv[8];
      row8(S.rawk, n, xk);
      row8(S.rawv, n, xv);
      ++nrows;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        unsigned h, l;
        fixed_split_biased(xk[i], h, l);
        kh[i] += h;
        kl[i] += l;
        fixed_split_biased(xv[i], h, l);
        vh[i] += h;
        vl[i] += l;
        exact &= fixed_split_exact<T>(xk[i]) && fixed_split_exact<T>(xv[i]);
        if (c0 + i < d) {
          mn[i] = fminf(mn[i], xv[i]);
          mx[i] = fmaxf(mx[i], xv[i]);
        }
        amax = fmaxf(amax, fmaxf(p.smooth_k ? fabsf(xk[i]) : 0.f, p.smooth_v ? fabsf(xv[i]) : 0.f));
      }
    }
    if (amax >= p.range_limit) record_error(p.err, kDevRange);
    long long ks[8], vs[8];
    const unsigned bias = static_cast<unsigned>(nrows) * static_cast<unsigned>(kRoundMagicBits);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ks[i] = (static_cast<long long>(static_cast<int>(kh[i] - bias)) << 20) + static_cast<int>(kl[i] - bias);
      vs[i] = (static_cast<long long>(static_cast<int>(vh[i] - bias)) << 20) + static_cast<int>(vl[i] - bias);
    }
    if (!exact) {
      // a bf16 value below 2^-17 or above 2^18: exact int64 conversions instead
#pragma unroll
      for (int i = 0; i < 8; ++i) ks[i] = vs[i] = 0;
      for (int n = rg; n < nk; n += RG) {
        float xk[8], xv[8];
        row8(S.rawk, n, xk);
        row8(S.rawv, n, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ks[i] += __float2ll_rz(xk[i] * 16777216.0f);
          vs[i] += __float2ll_rz(xv[i] * 16777216.0f);
        }
      }
    }
    // the row groups that share a warp (lanes with the same vec), then the 8 warps through
    // shared memory (the V^T and Q code space, written only later): shared-memory atomics on
    // the same 64 or 128 channels from every thread measured 17,000 cycles of this kernel's
    // 63,000 for 256 keys
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ks[i] += __shfl_xor_sync(0xffffffffu, ks[i], off);
        vs[i] += __shfl_xor_sync(0xffffffffu, vs[i], off);
        mn[i] = fminf(mn[i], __shfl_xor_sync(0xffffffffu, mn[i], off));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
      }
    }
    if (lane < TPR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        S.red_k[warp * DP + c0 + i] = ks[i];
        S.red_v[warp * DP + c0 + i] = vs[i];
        S.red_mn[warp * DP + c0 + i] = mn[i];
        S.red_mx[warp * DP + c0 + i] = mx[i];
      }
    }
  }
  __syncthreads();
  for (int c = t; c < DP; c += kSThreads) {
    float km = 0.f, vm = 0.f, vsc = 0.f, vr = 0.f;
    if (c < d) {
      long long ksum = 0, vsum = 0;
      float vmin = __int_as_float(0x7f800000), vmax = __int_as_float(0xff800000);
#pragma unroll
      for (int w = 0; w < kSThreads / 32; ++w) {
        ksum += S.red_k[w * DP + c];
        vsum += S.red_v[w * DP + c];
        vmin = fminf(vmin, S.red_mn[w * DP + c]);
        vmax = fmaxf(vmax, S.red_mx[w * DP + c]);
      }
      km = p.smooth_k ? fixed_point_mean(ksum, nk) : 0.f;
      vm = p.smooth_v ? fixed_point_mean(vsum, nk) : 0.f;
      const float hi = __fsub_rn(vmax, vm);
      const float lo = __fsub_rn(vmin, vm);
      const float a = fmaxf(fabsf(hi), fabsf(lo));
      vsc = a > 0.f ? __fdiv_rn(a, 448.0f) : 0.f;
      vr = a > 0.f ? __fdiv_rn(448.0f, a) : 0.f;
      if (kv_writer) {
        p.kmean[sidx + c] = km;
        p.vmean[sidx + c] = vm;
        p.vscale[sidx + c] = vsc;
        p.vrcp[sidx + c] = vr;
      }
    }
    S.kmean[c] = km;
    S.vmean[c] = vm;
    S.vscale[c] = vsc;
    S.vrcp[c] = vr;
  }
  __syncthreads();

  // ---- 2. K codes (groups of gk keys), V codes (per channel), Q codes (groups of gq rows)
  float kmean8[8], vmean8[8], vrcp8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    kmean8[i] = S.kmean[c0 + i];
    vmean8[i] = S.vmean[c0 + i];
    vrcp8[i] = S.vrcp[c0 + i];
  }
  // one pass over the key rows: the row maxima of |K - mean| and the V codes (rows of V^T in
  // slot order)
#pragma unroll 4
  for (int n = rg; n < nk_pad; n += RG) {
    float x[8], a = 0.f;
    uint8_t vcode[8];
    if (n < nk) {
      row8(S.rawk, n, x);
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, c0 + i < d ? fabsf(__fsub_rn(x[i], kmean8[i])) : 0.f);
      float xv[8];
      row8(S.rawv, n, xv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float vsm = c0 + i < d ? __fsub_rn(xv[i], vmean8[i]) : 0.f;
        vcode[i] = static_cast<uint8_t>(pack_e4m3x2(__fmul_rn(vsm, vrcp8[i]), 0.f) & 0xffu);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) vcode[i] = 0;
    }
    const int sl = v_slot(n);
#pragma unroll
    for (int i = 0; i < 8; ++i) S.vt8[(c0 + i) * S.nks + sl] = vcode[i];
#pragma unroll
    for (int off = 1; off < TPR; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    // the warp's rows (32 / TPR consecutive keys, within one K group: groups are 16 or 64
    // keys) to one value; |x| >= 0, so the float bits order like the values
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (lane == 0 && n < nk) atomicMax(&S.kgmax[n / p.gk], __float_as_uint(a));
  }
  __syncthreads();
  const int gk = p.gk, nkg = (nk + gk - 1) / gk;
  for (int g = t; g < nk_pad / 16; g += kSThreads) {
    const float a = __uint_as_float(S.kgmax[g]);  // 0 for groups past the keys
    S.gscale[g] = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
    S.grcp[g] = a > 0.f ? __fdiv_rn(127.0f, a) : 0.f;
    if (kv_writer && g < nkg) p.sk[plane_kv * p.sk_pp + g] = S.gscale[g];
  }
  const int gq = p.gq;
  for (int rr = t; rr < kSRows; rr += kSThreads) {
    const int g0 = rr / gq * gq;
    const float a = __uint_as_float(S.qgmax[rr / gq]);
    const float sc = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
    S.qscale[rr] = sc;
    S.qrcp[rr] = a > 0.f ? __fdiv_rn(127.0f, a) : 0.f;
    if (rr == g0 && r0 + rr < nq) p.sq[plane_q * p.sq_pp + (r0 + rr) / gq] = sc;
  }
  __syncthreads();
  // then the K codes, into the space of the raw V rows (the V codes are all written)
  if (kv_writer) {
    // V^T codes to the workspace in natural key order, 16 keys (one 16-byte store) at a time
    const int nchunk = (nk + 15) / 16;
    for (int it = t; it < DP * nchunk; it += kSThreads) {
      const int c = it / nchunk, n0 = (it - c * nchunk) * 16;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j >> 2] |= static_cast<uint32_t>(S.vt8[c * S.nks + v_slot(n0 + j)]) << (8 * (j & 3));
      *reinterpret_cast<uint4*>(p.vt + (plane_kv * p.dp + c) * p.vt_pitch + n0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
#pragma unroll 4
  for (int n = rg; n < nk_pad; n += RG) {
    __align__(16) __half kc16[8];
    if (n < nk) {
      float xk[8];
      row8(S.rawk, n, xk);
      const float rk = S.grcp[n / gk];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ks = c0 + i < d ? __fsub_rn(xk[i], kmean8[i]) : 0.f;
        kc16[i] = __int2half_rn(int8_code(ks, rk));
      }
      if (kv_writer)
        *reinterpret_cast<uint4*>(p.kc + (plane_kv * p.k_rows + n) * p.dp + c0) =
            *reinterpret_cast<const uint4*>(kc16);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) kc16[i] = __float2half_rn(0.f);
    }
    *reinterpret_cast<uint4*>(S.kcode + ((size_t)n * DP + ((vec ^ (n & 7)) << 3)) * 2) =
        *reinterpret_cast<const uint4*>(kc16);
  }
  const bool want_qkc = p.return_lse && p.smooth_k;
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int rr = rg + RG * u, i = r0 + rr;
    float x[8];
    unpack8<T>(qraw[u], x);
    float dot = 0.f;
    const float r = S.qrcp[rr];
    __align__(16) __half qc16[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qc16[j] = __int2half_rn(int8_code(x[j], r));
      dot = fmaf(x[j], kmean8[j], dot);
    }
    if (i < nq)
      *reinterpret_cast<uint4*>(p.qc + (plane_q * p.q_rows + i) * p.dp + c0) =
          *reinterpret_cast<const uint4*>(qc16);
    *reinterpret_cast<uint4*>(S.q16 + rr * DP + c0) = *reinterpret_cast<const uint4*>(qc16);
    if (want_qkc) {
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (vec == 0) S.qkt[rr] = dot;
    }
  }
  __syncthreads();

  // ---- 3. attention: warp w owns CTA rows 16 w .. 16 w + 15
  const int g = lane >> 2, q4 = lane & 3;
  const int ra = warp * 16 + g, rb = ra + 8;  // rows within the CTA
  const int ia = r0 + ra, ib = r0 + rb;       // query indices
  if (r0 + warp * 16 >= nq) return;           // warp-uniform; no block-wide sync follows
  uint32_t qa[DP / 16][4];  // A fragments of the Q codes, k-steps of 16 channels
#pragma unroll
  for (int ks = 0; ks < DP / 16; ++ks) {
    const int c = ks * 16 + q4 * 2;
    qa[ks][0] = *reinterpret_cast<const uint32_t*>(S.q16 + ra * DP + c);
    qa[ks][1] = *reinterpret_cast<const uint32_t*>(S.q16 + rb * DP + c);
    qa[ks][2] = *reinterpret_cast<const uint32_t*>(S.q16 + ra * DP + c + 8);
    qa[ks][3] = *reinterpret_cast<const uint32_t*>(S.q16 + rb * DP + c + 8);
  }
  const float sa = S.qscale[ra] * p.sm_scale * kSLog2e;
  const float sb = S.qscale[rb] * p.sm_scale * kSLog2e;
  float ma = __int_as_float(0xff800000), mb = ma;  // running maxima (log2 units)
  float la = 0.f, lb = 0.f;                        // this lane's share of the row sums
  float o[DP / 8][4];
#pragma unroll
  for (int nd = 0; nd < DP / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  const int lim_a = p.is_causal ? min(nk, ia + 1) : nk;
  const int lim_b = p.is_causal ? min(nk, ib + 1) : nk;
  const int kv_end = p.is_causal ? min(nk, r0 + warp * 16 + 16) : nk;
  const int lgk = p.lgk;
  // exact integer scores (in fp32) of 8-key column tile nt (absolute keys key0 + 8 nt ..)
  // for the warp's 16 rows; the K code rows are swizzled by 16-byte unit
  auto scores = [&](int key0, int nt, float (&sc)[4]) {
    sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
    const int key = key0 + nt * 8 + g;  // key & 7 == g
    const uint8_t* kr = S.kcode + (size_t)key * DP * 2 + q4 * 4;
#pragma unroll
    for (int ks = 0; ks < DP / 16; ++ks) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + (((2 * ks) ^ g) << 4));
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + (((2 * ks + 1) ^ g) << 4));
      mma_f16(sc, qa[ks], b0, b1);
    }
  };
  // head_dim 64: the tile's scores stay in registers between the max and the exponentials
  // (64 more registers); head_dim 128 computes them again for the exponentials (its Q
  // fragments and accumulators leave no room)
  constexpr bool kKeepScores = DP == 64;
  float scr[kKeepScores ? kSTile / 8 : 1][4];
  for (int kt = 0; kt * kSTile < kv_end; ++kt) {
    const int key0 = kt * kSTile;
    // maxima of the scaled scores over this tile's visible keys
    float ta = __int_as_float(0xff800000), tb = ta;
    if constexpr (kKeepScores) {
#pragma unroll
      for (int nt = 0; nt < kSTile / 8; ++nt) scores(key0, nt, scr[nt]);
    }
#pragma unroll(kKeepScores ? kSTile / 8 : 2)
    for (int nt = 0; nt < kSTile / 8; ++nt) {
      float sc[4];
      if constexpr (kKeepScores) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = scr[nt % (kSTile / 8)][e];
      } else {
        scores(key0, nt, sc);
      }
      const int j0 = key0 + nt * 8 + 2 * q4;
      const float cj = S.gscale[j0 >> lgk];
      const float ca = sa * cj, cb = sb * cj;
      if (j0 < lim_a) ta = fmaxf(ta, sc[0] * ca);
      if (j0 + 1 < lim_a) ta = fmaxf(ta, sc[1] * ca);
      if (j0 < lim_b) tb = fmaxf(tb, sc[2] * cb);
      if (j0 + 1 < lim_b) tb = fmaxf(tb, sc[3] * cb);
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      ta = fmaxf(ta, __shfl_xor_sync(0xffffffffu, ta, off));
      tb = fmaxf(tb, __shfl_xor_sync(0xffffffffu, tb, off));
    }
    const float na = fmaxf(ma, ta), nb = fmaxf(mb, tb);
    const float ua = na == __int_as_float(0xff800000) ? 0.f : na;
    const float ub = nb == __int_as_float(0xff800000) ? 0.f : nb;
    const float alpha_a = ex2s(ma - ua), alpha_b = ex2s(mb - ub);
    const float bias_a = kSLog2Sigma - ua, bias_b = kSLog2Sigma - ub;
    la *= alpha_a;
    lb *= alpha_b;
#pragma unroll
    for (int nd = 0; nd < DP / 8; ++nd) {
      o[nd][0] *= alpha_a;
      o[nd][1] *= alpha_a;
      o[nd][2] *= alpha_b;
      o[nd][3] *= alpha_b;
    }
    ma = na;
    mb = nb;
    // P~ per 32-key chunk as an A fragment, then P~ V
#pragma unroll(kKeepScores ? kSTile / 32 : 1)
    for (int kc = 0; kc < kSTile / 32; ++kc) {
      uint32_t pa[4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t wa = 0, wb = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int nt = kc * 4 + half * 2 + u;
          float sc[4];
          if constexpr (kKeepScores) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[e] = scr[nt % (kSTile / 8)][e];
          } else {
            scores(key0, nt, sc);
          }
          const int j0 = key0 + nt * 8 + 2 * q4;
          const float cj = S.gscale[j0 >> lgk];
          const float ca = sa * cj, cb = sb * cj;
          const float e0 = j0 < lim_a ? ex2s(fmaf(sc[0], ca, bias_a)) : 0.f;
          const float e1 = j0 + 1 < lim_a ? ex2s(fmaf(sc[1], ca, bias_a)) : 0.f;
          const float e2 = j0 < lim_b ? ex2s(fmaf(sc[2], cb, bias_b)) : 0.f;
          const float e3 = j0 + 1 < lim_b ? ex2s(fmaf(sc[3], cb, bias_b)) : 0.f;
          la += e0 + e1;
          lb += e2 + e3;
          wa |= pack_e4m3x2(e0, e1) << (16 * u);
          wb |= pack_e4m3x2(e2, e3) << (16 * u);
        }
        pa[2 * half] = wa;      // row g: slots 4 q .. (+16 for the second half)
        pa[2 * half + 1] = wb;  // row g + 8
      }
#pragma unroll
      for (int nd = 0; nd < DP / 8; ++nd) {
        const uint8_t* vr = S.vt8 + (nd * 8 + g) * S.nks + key0 + kc * 32 + q4 * 4;
        mma_e4m3(o[nd], pa, *reinterpret_cast<const uint32_t*>(vr),
                 *reinterpret_cast<const uint32_t*>(vr + 16));
      }
    }
  }
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    la += __shfl_xor_sync(0xffffffffu, la, off);
    lb += __shfl_xor_sync(0xffffffffu, lb, off);
  }
  const float inv_a = 1.0f / la, inv_b = 1.0f / lb;
  uint16_t* const oa = static_cast<uint16_t*>(p.o) + (int64_t)b * p.o_sb + (int64_t)ia * p.o_sn + (int64_t)h * p.o_sh;
  uint16_t* const ob = static_cast<uint16_t*>(p.o) + (int64_t)b * p.o_sb + (int64_t)ib * p.o_sn + (int64_t)h * p.o_sh;
#pragma unroll
  for (int nd = 0; nd < DP / 8; ++nd) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = nd * 8 + 2 * q4 + e;
      if (c < d) {
        const float vs = S.vscale[c], vm = S.vmean[c];
        if (ia < nq) {
          const float v = fmaf(o[nd][e] * vs, inv_a, vm);
          oa[c] = p.dtype == 0 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
        if (ib < nq) {
          const float v = fmaf(o[nd][2 + e] * vs, inv_b, vm);
          ob[c] = p.dtype == 0 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
      }
    }
  }
  if (p.return_lse && q4 == 0) {
    const float qka = want_qkc ? S.qkt[ra] : 0.f, qkb = want_qkc ? S.qkt[rb] : 0.f;
    if (ia < nq)
      p.lse[plane_q * p.nq + ia] = (ma + __log2f(la) - kSLog2Sigma) * 0.6931471805599453f + p.sm_scale * qka;
    if (ib < nq)
      p.lse[plane_q * p.nq + ib] = (mb + __log2f(lb) - kSLog2Sigma) * 0.6931471805599453f + p.sm_scale * qkb;
  }
}

// Clears the call's status words; lets the short kernel's launch start at once.
__global__ void short_status_clear(int* err, int n) {
  pdl_trigger();
  for (int i = threadIdx.x; i < n; i += blockDim.x) err[i] = 0;
}

template <typename T, int DP>
cudaError_t launch_short_t(const Problem& p, cudaStream_t st) {
  const int nk_pad = (p.nk + kSTile - 1) / kSTile * kSTile;
  const size_t smem = short_offsets(DP, nk_pad).total;
  static std::atomic<int> limits[64];
  const cudaError_t e = raise_smem_limit(short_attn_kernel<T, DP>, (int)smem, limits);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.nq + kSRows - 1) / kSRows, p.hq, p.batch);
  const cudaError_t el = launch_pdl(short_attn_kernel<T, DP>, grid, dim3(kSThreads), smem, st, p);
  return el != cudaSuccess ? el : cudaGetLastError();
}

}  // namespace

cudaError_t launch_short_status_clear(int* err, int words, cudaStream_t st) {
  short_status_clear<<<1, 32, 0, st>>>(err, words);
  return cudaGetLastError();
}

cudaError_t launch_short_attention(const Problem& p, cudaStream_t st) {
  if (p.dtype == 0)
    return p.dp == 64 ? launch_short_t<__half, 64>(p, st) : launch_short_t<__half, 128>(p, st);
  return p.dp == 64 ? launch_short_t<__nv_bfloat16, 64>(p, st) : launch_short_t<__nv_bfloat16, 128>(p, st);
}

}  // namespace sage
