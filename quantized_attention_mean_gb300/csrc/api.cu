// Host side of the C ABI declared in include/sageattn.h: argument validation, workspace
// carving, TMA tensor maps and the launch sequence. No device memory is allocated here.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/sageattn.h"
#include "launch.h"

namespace sage {
namespace {

// ------------------------------------------------------------------------------ workspace
constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

const int kQGroup[3] = {128, 32, 1};   // per_block, per_warp, per_thread
const int kKGroup[3] = {64, 64, 16};

struct Layout {
  size_t off_err, off_ksum, off_vsum, off_vmin, off_vmax, off_kmean, off_vmean, off_vscale, off_vrcp,
      off_qc, off_kc, off_vt, off_sq, off_sk, off_qkc, off_seqinfo, total;
  int64_t q_rows, k_rows, vt_pitch, sq_pp, sk_pp, planes_q, planes_kv, n_stats;
  int dp, gq, gk;
};

// Dense: planes are (batch, head) pairs with exactly seqlen rows each. Varlen: planes are
// heads; each sequence owns a 128-row aligned segment of the plane, so a plane has at most
// total + 128 * batch rows.
bool make_layout(bool varlen, int batch, int hq, int hkv, int64_t lq, int64_t lk, int d, int gran,
                 Layout* L) {
  if (batch < 0 || hq < 1 || hkv < 1 || lq < 0 || lk < 0 || d < 1 || d > 128 || gran < 0 ||
      gran > 2)
    return false;
  L->dp = d <= 64 ? 64 : 128;
  L->gq = kQGroup[gran];
  L->gk = kKGroup[gran];
  if (varlen) {
    L->planes_q = hq;
    L->planes_kv = hkv;
    L->q_rows = round_up(lq, 128) + 128 * (int64_t)batch;
    L->k_rows = round_up(lk, 128) + 128 * (int64_t)batch;
    L->vt_pitch = L->k_rows;
  } else {
    L->planes_q = (int64_t)batch * hq;
    L->planes_kv = (int64_t)batch * hkv;
    L->q_rows = lq;
    L->k_rows = lk;
    L->vt_pitch = round_up(lk, 16);
  }
  L->sq_pp = (L->q_rows + L->gq - 1) / L->gq;
  L->sk_pp = (L->k_rows + L->gk - 1) / L->gk;
  L->n_stats = (int64_t)batch * hkv * d;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += align_up(bytes); return at; };
  L->off_err = take(16);
  L->off_ksum = take(8 * L->n_stats);
  L->off_vsum = take(8 * L->n_stats);
  L->off_vmin = take(4 * L->n_stats);
  L->off_vmax = take(4 * L->n_stats);
  L->off_kmean = take(4 * L->n_stats);
  L->off_vmean = take(4 * L->n_stats);
  L->off_vscale = take(4 * L->n_stats);
  L->off_vrcp = take(4 * L->n_stats);
  L->off_qc = take(2 * (size_t)L->planes_q * L->q_rows * L->dp);
  L->off_kc = take(2 * (size_t)L->planes_kv * L->k_rows * L->dp);
  // V^T: E4M3 bytes, or fp16 for the FP16 P·V variant (two bytes reserved per element)
  L->off_vt = take((size_t)L->planes_kv * L->dp * L->vt_pitch * 2);
  L->off_sq = take(4 * (size_t)L->planes_q * L->sq_pp);
  L->off_sk = take(4 * (size_t)L->planes_kv * L->sk_pp);
  L->off_qkc = take(4 * (size_t)L->planes_q * L->q_rows);
  L->off_seqinfo = take(4 * (size_t)kSiRows * (varlen ? batch : 0));
  L->total = o;
  return true;
}

void carve(Problem& p, const Layout& L, void* ws) {
  char* w = static_cast<char*>(ws);
  p.err = reinterpret_cast<int*>(w + L.off_err);
  p.ksum = reinterpret_cast<long long*>(w + L.off_ksum);
  p.vsum = reinterpret_cast<long long*>(w + L.off_vsum);
  p.vmin = reinterpret_cast<unsigned*>(w + L.off_vmin);
  p.vmax = reinterpret_cast<unsigned*>(w + L.off_vmax);
  p.kmean = reinterpret_cast<float*>(w + L.off_kmean);
  p.vmean = reinterpret_cast<float*>(w + L.off_vmean);
  p.vscale = reinterpret_cast<float*>(w + L.off_vscale);
  p.vrcp = reinterpret_cast<float*>(w + L.off_vrcp);
  p.qc = reinterpret_cast<__half*>(w + L.off_qc);
  p.kc = reinterpret_cast<__half*>(w + L.off_kc);
  p.vt = reinterpret_cast<uint8_t*>(w + L.off_vt);
  p.sq = reinterpret_cast<float*>(w + L.off_sq);
  p.sk = reinterpret_cast<float*>(w + L.off_sk);
  p.qkc = reinterpret_cast<float*>(w + L.off_qkc);
  p.seqinfo = reinterpret_cast<int*>(w + L.off_seqinfo);
  p.q_rows = L.q_rows;
  p.k_rows = L.k_rows;
  p.vt_pitch = L.vt_pitch;
  p.sq_pp = L.sq_pp;
  p.sk_pp = L.sk_pp;
  p.dp = L.dp;
  p.gq = L.gq;
  p.gk = L.gk;
  p.lgk = L.gk == 16 ? 4 : 6;
}

// ------------------------------------------------------------------------------ device info
int g_dev_ok[64];  // 0 unknown, 1 sm_103, 2 other
int g_stall = 0;   // test hook (sage_debug_stall_attention)
int g_path = 0;    // sage_debug_select_path: 0 / 1 main pipeline, 2 short kernel where it fits
long long* g_trace = nullptr;  // sage_debug_trace_attention
std::mutex g_mu;

bool device_is_sm103() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev_ok[dev]) return g_dev_ok[dev] == 1;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  const bool ok = major == 10 && minor == 3;
  std::lock_guard<std::mutex> lk(g_mu);
  g_dev_ok[dev] = ok ? 1 : 2;
  return ok;
}

// ------------------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-d tiled map with a 128-byte swizzle: dims (inner, rows, planes), byte strides of rows
// and planes, box (inner_box, rows_box, 1).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
              uint64_t planes, uint64_t row_bytes, uint64_t plane_bytes, uint32_t box_inner,
              uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {row_bytes, plane_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------ validation
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Common {
  int hq, hkv, d, dtype, is_causal, return_lse, gran, acc, smooth_k, smooth_v;
  float sm_scale;
};

int check_common(const Common& c, const float* lse) {
  if (c.d < 1 || c.d > 128) return SAGE_ERR_HEAD_DIM;
  if (c.dtype != SAGE_F16 && c.dtype != SAGE_BF16) return SAGE_ERR_DTYPE;
  if (c.hq < 1 || c.hkv < 1) return SAGE_ERR_INVALID_ARG;
  if (c.hq % c.hkv) return SAGE_ERR_GQA;
  if (c.gran < SAGE_PER_BLOCK || c.gran > SAGE_PER_THREAD) return SAGE_ERR_INVALID_ARG;
  if (c.acc == SAGE_ACC_FP16) return SAGE_ERR_UNSUPPORTED;
  if (c.acc < SAGE_ACC_FP32 || c.acc > SAGE_ACC_FP16) return SAGE_ERR_INVALID_ARG;
  if (c.return_lse && (lse == nullptr || !aligned(lse, 4))) return SAGE_ERR_INVALID_ARG;
  return SAGE_OK;
}

void fill_common(Problem& p, const Common& c) {
  p.hq = c.hq; p.hkv = c.hkv; p.d = c.d; p.dtype = c.dtype;
  p.is_causal = c.is_causal ? 1 : 0;
  p.return_lse = c.return_lse ? 1 : 0;
  p.smooth_k = c.smooth_k ? 1 : 0;
  p.smooth_v = c.smooth_v ? 1 : 0;
  p.sm_scale = (std::isnan(c.sm_scale) || c.sm_scale <= 0.f)
                   ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.d)))
                   : c.sm_scale;
}

// Smallest float >= 2^38 / n (the fixed-point mean's magnitude limit).
float range_limit(int64_t n) {
  const double thr = 274877906944.0 / static_cast<double>(n > 0 ? n : 1);
  float f = static_cast<float>(thr);
  if (static_cast<double>(f) < thr) f = std::nextafter(f, INFINITY);
  return f;
}

// ------------------------------------------------------------------------------ profiling
struct StageEvents { cudaEvent_t e[4]; };
constexpr int kMaxProfiled = 8192;
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<StageEvents> g_prof_pool;  // created on enable, reused
int g_prof_used = 0;

// Returns the event set for this call, or nullptr when profiling is off / the record is full.
StageEvents* prof_next() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || g_prof_used >= (int)g_prof_pool.size()) return nullptr;
  return &g_prof_pool[g_prof_used++];
}

thread_local char g_last_err[192] = "no error";

// Records a failed CUDA call for sage_last_cuda_error and returns SAGE_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_err, sizeof(g_last_err), "%s: %s (%s)", where, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return SAGE_ERR_CUDA;
}

int run_pipeline(Problem& p, const Layout& L, int max_len_q, int max_len_k, cudaStream_t st) {
  CUtensorMap maps[3];
  const uint64_t dp = static_cast<uint64_t>(L.dp);
  bool ok = make_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.qc, dp, L.q_rows, L.planes_q,
                     dp * 2, dp * 2 * L.q_rows, 64, 128) &&
            make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.kc, dp, L.k_rows, L.planes_kv,
                     dp * 2, dp * 2 * L.k_rows, 64, 128) &&
            (p.pv16 ? make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.vt,
                               p.varlen ? L.k_rows : static_cast<uint64_t>(p.nk), dp, L.planes_kv,
                               L.vt_pitch * 2, L.vt_pitch * 2 * dp, 64, L.dp)
                    : make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.vt,
                               p.varlen ? L.k_rows : static_cast<uint64_t>(p.nk), dp, L.planes_kv,
                               L.vt_pitch, L.vt_pitch * dp, 128, L.dp));
  if (!ok) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  StageEvents* ev = prof_next();
  auto mark = [&](int i) { if (ev) cudaEventRecord(ev->e[i], st); };
  cudaError_t e;
  mark(0);
  // status and statistics accumulators (contiguous from off_err up to off_kmean): one clear
  if ((e = cudaMemsetAsync(p.err, 0, L.off_kmean - L.off_err, st)) != cudaSuccess)
    return cuda_fail(e, "status and statistics reset");
  if (p.varlen && (e = launch_varlen_setup(p, st)) != cudaSuccess) return cuda_fail(e, "varlen set-up");
  if ((e = launch_kv_stats(p, max_len_k, st)) != cudaSuccess) return cuda_fail(e, "K/V statistics");
  if ((e = launch_finalize(p, static_cast<int>(L.n_stats), st)) != cudaSuccess) return cuda_fail(e, "statistics finalize");
  mark(1);
  if ((e = launch_quant(p, max_len_q, max_len_k, st)) != cudaSuccess) return cuda_fail(e, "quantisation");
  mark(2);
  const int pairs = (max_len_q + 2 * kTileRows - 1) / (2 * kTileRows);
  if ((e = launch_attention(p, maps, pairs, st)) != cudaSuccess) return cuda_fail(e, "attention");
  mark(3);
  return SAGE_OK;
}

// One launch (after a clear of the status word) for problems the short-sequence kernel takes.
int run_short(Problem& p, const Layout& L, cudaStream_t st) {
  StageEvents* ev = prof_next();
  auto mark = [&](int i) { if (ev) cudaEventRecord(ev->e[i], st); };
  cudaError_t e;
  mark(0);
  // a one-thread clear kernel rather than a memset, so that the short kernel (launched as a
  // programmatic dependent) starts while it finishes
  if ((e = launch_short_status_clear(p.err, static_cast<int>((L.off_ksum - L.off_err) / 4), st)) != cudaSuccess)
    return cuda_fail(e, "status reset");
  mark(1);
  mark(2);
  if ((e = launch_short_attention(p, st)) != cudaSuccess) return cuda_fail(e, "short attention");
  mark(3);
  return SAGE_OK;
}

int dense_impl(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
               const sage_tensor* out, float* lse, int batch, int hq, int hkv, int nq, int nk,
               int d, int dtype, int layout, int is_causal, float sm_scale, int return_lse,
               int gran, int acc, int smooth_k, int smooth_v, void* ws, size_t ws_bytes,
               int32_t* dbg_scores, void* stream, int pv = 0) {
  if (!q || !k || !v || !out) return SAGE_ERR_INVALID_ARG;
  const Common c{hq, hkv, d, dtype, is_causal, return_lse, gran, acc, smooth_k, smooth_v, sm_scale};
  int st = check_common(c, lse);
  if (st != SAGE_OK) return st;
  if (layout != SAGE_HND && layout != SAGE_NHD) return SAGE_ERR_INVALID_ARG;
  if (batch < 0 || nq < 0 || nk < 0) return SAGE_ERR_INVALID_ARG;
  if (batch == 0 || nq == 0) return SAGE_OK;
  if (nk == 0) return SAGE_ERR_INVALID_ARG;
  if (!q->data || !k->data || !v->data || !out->data) return SAGE_ERR_INVALID_ARG;
  const sage_tensor* ts[4] = {q, k, v, out};
  bool vec16 = d % 8 == 0;
  for (const sage_tensor* t : ts) {
    if (!aligned(t->data, 2)) return SAGE_ERR_STRIDE;
    for (int i = 0; i < 3; ++i)
      if (t->stride[i] < 0) return SAGE_ERR_STRIDE;
    vec16 = vec16 && aligned(t->data, 16) && t->stride[0] % 8 == 0 && t->stride[1] % 8 == 0 &&
            t->stride[2] % 8 == 0;
  }
  Layout L;
  if (!make_layout(false, batch, hq, hkv, nq, nk, d, gran, &L)) return SAGE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < L.total) return SAGE_ERR_WORKSPACE;
  if (!device_is_sm103()) return SAGE_ERR_DEVICE;
  Problem p;
  std::memset(&p, 0, sizeof(p));
  fill_common(p, c);
  p.batch = batch; p.nq = nq; p.nk = nk; p.varlen = 0; p.vec16 = vec16 ? 1 : 0;
  p.pv16 = pv != 0;  // 1: FP16 P·V variant, 2: FP4 microscaled variant (both on fp16 operands)
  p.fp4 = pv == 2;
  // Attention CTAs pairs-fastest when the non-causal problem's K / V codes exceed half the 129 MB
  // L2: the resident CTAs then share one or two heads' K / V instead of re-reading every head's
  // from DRAM (measured on the 2x48x17776 head_dim 64 shape: 8.795 ms vs 8.839; on 2x8x4096
  // head_dim 128, whose K / V fit in L2, heads fastest stays faster: 0.1238 vs 0.1252 ms)
  {
    const double kv_bytes = (double)batch * hkv * nk * (d <= 64 ? 64 : 128) * 3.0;
    p.pair_major = (!is_causal && kv_bytes > 64.0 * 1024 * 1024) ? 1 : 0;
  }
  // element strides (b, h, n) from the layout's dimension order
  auto bhn = [layout](const sage_tensor* t, int64_t& sb, int64_t& sh, int64_t& sn) {
    sb = t->stride[0];
    if (layout == SAGE_HND) { sh = t->stride[1]; sn = t->stride[2]; }
    else { sn = t->stride[1]; sh = t->stride[2]; }
  };
  p.q = q->data; bhn(q, p.q_sb, p.q_sh, p.q_sn);
  p.k = k->data; bhn(k, p.k_sb, p.k_sh, p.k_sn);
  p.v = v->data; bhn(v, p.v_sb, p.v_sh, p.v_sn);
  p.o = out->data; bhn(out, p.o_sb, p.o_sh, p.o_sn);
  p.lse = lse;
  p.range_limit = range_limit(nk);
  p.dbg_scores = dbg_scores;
  p.dbg_stall = g_stall;
  p.dbg_trace = g_trace;
  carve(p, L, ws);
  // The one-launch short-sequence kernel can take a problem that fits it (the score dump,
  // trace and stall hooks belong to the main pipeline's kernels, and the FP16 P·V and FP4
  // variants have no short form). By default it takes the head_dim-64 problems called
  // directly: measured per call at 256^2, head_dim 64, 28.4 us against 36.8 for the four
  // launches, and at 1024 x 256 (16 heads) 28.2 against 36.8. Into a CUDA graph being captured
  // the four launches go instead (replayed they measured 21.7 us against 26.7), and at
  // head_dim 128 always (52 us against 36 direct, 22 replayed).
  const bool short_ok = pv == 0 && !dbg_scores && !g_trace && !g_stall && nk <= kShortMaxKeys &&
                        nq <= kShortMaxQueries;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (short_ok && g_path == 2) return run_short(p, L, cs);
  if (short_ok && g_path == 0 && p.dp == 64) {
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusActive;
    if (cudaStreamIsCapturing(cs, &capture) != cudaSuccess) {
      cudaGetLastError();  // unknown: take the pipeline, which captures either way
      capture = cudaStreamCaptureStatusActive;
    }
    if (capture == cudaStreamCaptureStatusNone) return run_short(p, L, cs);
  }
  return run_pipeline(p, L, nq, nk, cs);
}

}  // namespace

int note_cuda_failure(cudaError_t e, const char* where) { return cuda_fail(e, where); }

}  // namespace sage

using namespace sage;

extern "C" {

size_t sage_attn_workspace_size(int batch, int heads_q, int heads_kv, int seqlen_q, int seqlen_k,
                                int head_dim, int qk_quant_gran) {
  Layout L;
  if (!make_layout(false, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim, qk_quant_gran, &L))
    return 0;
  return L.total;
}

int sage_attn(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
              const sage_tensor* out, float* lse, int batch, int heads_q, int heads_kv,
              int seqlen_q, int seqlen_k, int head_dim, int dtype, int tensor_layout, int is_causal,
              float sm_scale, int return_lse, int qk_quant_gran, int pv_accum_dtype, int smooth_k,
              int smooth_v, void* workspace, size_t workspace_bytes, void* stream) {
  return dense_impl(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim,
                    dtype, tensor_layout, is_causal, sm_scale, return_lse, qk_quant_gran,
                    pv_accum_dtype, smooth_k, smooth_v, workspace, workspace_bytes, nullptr,
                    stream);
}

int sage_attn_qk_int8_pv_fp16(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                              const sage_tensor* out, float* lse, int batch, int heads_q,
                              int heads_kv, int seqlen_q, int seqlen_k, int head_dim, int dtype,
                              int tensor_layout, int is_causal, float sm_scale, int return_lse,
                              int qk_quant_gran, int pv_accum_dtype, int smooth_k, int smooth_v,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return dense_impl(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim,
                    dtype, tensor_layout, is_causal, sm_scale, return_lse, qk_quant_gran,
                    pv_accum_dtype, smooth_k, smooth_v, workspace, workspace_bytes, nullptr,
                    stream, 1);
}

int sage_attn_fp4(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                  const sage_tensor* out, float* lse, int batch, int heads_q, int heads_kv,
                  int seqlen_q, int seqlen_k, int head_dim, int dtype, int tensor_layout,
                  int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
                  int pv_accum_dtype, int smooth_k, int smooth_v, void* workspace,
                  size_t workspace_bytes, void* stream) {
  return dense_impl(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim,
                    dtype, tensor_layout, is_causal, sm_scale, return_lse, qk_quant_gran,
                    pv_accum_dtype, smooth_k, smooth_v, workspace, workspace_bytes, nullptr,
                    stream, 2);
}

int sage_attn_debug_scores(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                           const sage_tensor* out, float* lse, int batch, int heads_q,
                           int heads_kv, int seqlen_q, int seqlen_k, int head_dim, int dtype,
                           int tensor_layout, int is_causal, float sm_scale, int return_lse,
                           int qk_quant_gran, int pv_accum_dtype, int smooth_k, int smooth_v,
                           void* workspace, size_t workspace_bytes, int32_t* scores,
                           void* stream) {
  if (!scores || !aligned(scores, 4)) return SAGE_ERR_INVALID_ARG;
  return dense_impl(q, k, v, out, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim,
                    dtype, tensor_layout, is_causal, sm_scale, return_lse, qk_quant_gran,
                    pv_accum_dtype, smooth_k, smooth_v, workspace, workspace_bytes, scores,
                    stream);
}

size_t sage_attn_varlen_workspace_size(int batch, int heads_q, int heads_kv, int total_q,
                                       int total_k, int head_dim, int qk_quant_gran) {
  Layout L;
  if (!make_layout(true, batch, heads_q, heads_kv, total_q, total_k, head_dim, qk_quant_gran, &L))
    return 0;
  return L.total;
}

static int varlen_impl(const sage_packed* q, const sage_packed* k, const sage_packed* v,
                       const sage_packed* out, float* lse, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int batch, int max_seqlen_q, int max_seqlen_k,
                       int total_q, int total_k, int heads_q, int heads_kv, int head_dim, int dtype,
                       int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
                       int pv_accum_dtype, int smooth_k, int smooth_v, void* workspace,
                       size_t workspace_bytes, void* stream, int pv16) {
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return SAGE_ERR_INVALID_ARG;
  const Common c{heads_q, heads_kv, head_dim, dtype, is_causal, return_lse, qk_quant_gran,
                 pv_accum_dtype, smooth_k, smooth_v, sm_scale};
  int st = check_common(c, lse);
  if (st != SAGE_OK) return st;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return SAGE_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0) return SAGE_OK;
  if (total_k == 0 || max_seqlen_k == 0) return SAGE_ERR_INVALID_ARG;
  if (!cu_seqlens_q || !cu_seqlens_k || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return SAGE_ERR_INVALID_ARG;
  const sage_packed* ts[4] = {q, k, v, out};
  bool vec16 = head_dim % 8 == 0;
  for (const sage_packed* t : ts) {
    if (!t->data) return SAGE_ERR_INVALID_ARG;
    if (!aligned(t->data, 2) || t->stride_token < 0 || t->stride_head < 0) return SAGE_ERR_STRIDE;
    vec16 = vec16 && aligned(t->data, 16) && t->stride_token % 8 == 0 && t->stride_head % 8 == 0;
  }
  Layout L;
  if (!make_layout(true, batch, heads_q, heads_kv, total_q, total_k, head_dim, qk_quant_gran, &L))
    return SAGE_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total)
    return SAGE_ERR_WORKSPACE;
  if (!device_is_sm103()) return SAGE_ERR_DEVICE;
  Problem p;
  std::memset(&p, 0, sizeof(p));
  fill_common(p, c);
  p.batch = batch; p.nq = max_seqlen_q; p.nk = max_seqlen_k; p.varlen = 1;
  p.vec16 = vec16 ? 1 : 0;
  p.pv16 = pv16;
  p.total_q = total_q; p.total_k = total_k;
  p.cu_q = cu_seqlens_q; p.cu_k = cu_seqlens_k;
  p.q = q->data; p.q_sb = 0; p.q_sn = q->stride_token; p.q_sh = q->stride_head;
  p.k = k->data; p.k_sb = 0; p.k_sn = k->stride_token; p.k_sh = k->stride_head;
  p.v = v->data; p.v_sb = 0; p.v_sn = v->stride_token; p.v_sh = v->stride_head;
  p.o = out->data; p.o_sb = 0; p.o_sn = out->stride_token; p.o_sh = out->stride_head;
  p.lse = lse;
  p.lse_plane = total_q;
  p.range_limit = 0.f;  // per sequence on the device
  p.dbg_stall = g_stall;
  carve(p, L, workspace);
  return run_pipeline(p, L, max_seqlen_q, max_seqlen_k, static_cast<cudaStream_t>(stream));
}

int sage_attn_varlen(const sage_packed* q, const sage_packed* k, const sage_packed* v,
                     const sage_packed* out, float* lse, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_k, int batch, int max_seqlen_q, int max_seqlen_k,
                     int total_q, int total_k, int heads_q, int heads_kv, int head_dim, int dtype,
                     int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
                     int pv_accum_dtype, int smooth_k, int smooth_v, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return varlen_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q,
                     max_seqlen_k, total_q, total_k, heads_q, heads_kv, head_dim, dtype, is_causal,
                     sm_scale, return_lse, qk_quant_gran, pv_accum_dtype, smooth_k, smooth_v,
                     workspace, workspace_bytes, stream, 0);
}

int sage_attn_varlen_qk_int8_pv_fp16(const sage_packed* q, const sage_packed* k,
                                     const sage_packed* v, const sage_packed* out, float* lse,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                                     int total_k, int heads_q, int heads_kv, int head_dim,
                                     int dtype, int is_causal, float sm_scale, int return_lse,
                                     int qk_quant_gran, int pv_accum_dtype, int smooth_k,
                                     int smooth_v, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return varlen_impl(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q,
                     max_seqlen_k, total_q, total_k, heads_q, heads_kv, head_dim, dtype, is_causal,
                     sm_scale, return_lse, qk_quant_gran, pv_accum_dtype, smooth_k, smooth_v,
                     workspace, workspace_bytes, stream, 1);
}

const char* sage_status_string(int status) {
  switch (status) {
    case SAGE_OK: return "SAGE_OK";
    case SAGE_ERR_INVALID_ARG: return "SAGE_ERR_INVALID_ARG: invalid argument";
    case SAGE_ERR_HEAD_DIM: return "SAGE_ERR_HEAD_DIM: head_dim must be in [1, 128]";
    case SAGE_ERR_DTYPE: return "SAGE_ERR_DTYPE: dtype must be fp16 or bf16";
    case SAGE_ERR_STRIDE: return "SAGE_ERR_STRIDE: misaligned pointer or unsupported stride";
    case SAGE_ERR_GQA: return "SAGE_ERR_GQA: query heads must be a multiple of KV heads";
    case SAGE_ERR_WORKSPACE: return "SAGE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SAGE_ERR_RANGE: return "SAGE_ERR_RANGE: input magnitude too large for the exact mean";
    case SAGE_ERR_UNSUPPORTED: return "SAGE_ERR_UNSUPPORTED: pure fp16 P.V accumulation is not supported";
    case SAGE_ERR_TIMEOUT: return "SAGE_ERR_TIMEOUT: a bounded device wait expired";
    case SAGE_ERR_CUDA: return "SAGE_ERR_CUDA: a CUDA call failed";
    case SAGE_ERR_DEVICE: return "SAGE_ERR_DEVICE: device is not compute capability 10.3";
    case SAGE_ERR_SEQLENS: return "SAGE_ERR_SEQLENS: invalid cu_seqlens";
    default: return "unknown sage_status";
  }
}

const char* sage_last_cuda_error(void) { return g_last_err; }

int sage_read_device_status(const void* workspace, void* stream) {
  if (!workspace) return SAGE_ERR_INVALID_ARG;
  int v = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SAGE_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SAGE_ERR_CUDA;
  return v;
}

int sage_device_supported(void) { return device_is_sm103() ? 1 : 0; }

int sage_debug_export_quant(const void* workspace, int batch, int heads_q, int heads_kv,
                            int seqlen_q, int seqlen_k, int head_dim, int qk_quant_gran,
                            int8_t* q8, float* sq, int8_t* k8, float* sk, float* kmean,
                            float* vmean, float* vscale, uint8_t* v8, void* stream) {
  Layout L;
  if (!workspace ||
      !make_layout(false, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim, qk_quant_gran, &L))
    return SAGE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(workspace);
  const int pq = static_cast<int>(L.planes_q), pk = static_cast<int>(L.planes_kv);
  bool ok = true;
  if (q8) ok &= launch_export_codes(reinterpret_cast<const __half*>(w + L.off_qc), L.q_rows, L.dp,
                                    head_dim, pq, seqlen_q, q8, st) == cudaSuccess;
  if (k8) ok &= launch_export_codes(reinterpret_cast<const __half*>(w + L.off_kc), L.k_rows, L.dp,
                                    head_dim, pk, seqlen_k, k8, st) == cudaSuccess;
  if (v8) ok &= launch_export_vt(reinterpret_cast<const uint8_t*>(w + L.off_vt), L.vt_pitch, L.dp,
                                 head_dim, pk, seqlen_k, v8, st) == cudaSuccess;
  auto copy = [&](void* dst, size_t off, size_t bytes) {
    if (dst) ok &= cudaMemcpyAsync(dst, w + off, bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  };
  copy(sq, L.off_sq, 4 * (size_t)L.planes_q * L.sq_pp);
  copy(sk, L.off_sk, 4 * (size_t)L.planes_kv * L.sk_pp);
  copy(kmean, L.off_kmean, 4 * (size_t)L.n_stats);
  copy(vmean, L.off_vmean, 4 * (size_t)L.n_stats);
  copy(vscale, L.off_vscale, 4 * (size_t)L.n_stats);
  return ok ? SAGE_OK : SAGE_ERR_CUDA;
}

int sage_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on && g_prof_pool.empty()) {
    g_prof_pool.resize(kMaxProfiled);
    for (auto& se : g_prof_pool)
      for (auto& e : se.e)
        if (cudaEventCreate(&e) != cudaSuccess) return SAGE_ERR_CUDA;
  }
  g_prof_on = on != 0;
  g_prof_used = 0;
  return SAGE_OK;
}

int sage_profile_read(double* stage_ms, int* calls) {
  if (!stage_ms || !calls) return SAGE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  stage_ms[0] = stage_ms[1] = stage_ms[2] = 0.0;
  for (int c = 0; c < g_prof_used; ++c) {
    StageEvents& se = g_prof_pool[c];
    if (cudaEventSynchronize(se.e[3]) != cudaSuccess) return SAGE_ERR_CUDA;
    for (int i = 0; i < 3; ++i) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, se.e[i], se.e[i + 1]) != cudaSuccess) return SAGE_ERR_CUDA;
      stage_ms[i] += ms;
    }
  }
  *calls = g_prof_used;
  g_prof_used = 0;
  return SAGE_OK;
}

int sage_debug_trace_attention(long long* clocks) {
  g_trace = clocks;
  return SAGE_OK;
}

int sage_debug_select_path(int path) {
  if (path < 0 || path > 2) return SAGE_ERR_INVALID_ARG;
  g_path = path;
  return SAGE_OK;
}

int sage_debug_stall_attention(int on) {
  g_stall = on ? 1 : 0;
  return SAGE_OK;
}

int sage_debug_e2m1(const float* x, uint8_t* out, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !out))) return SAGE_ERR_INVALID_ARG;
  if (n == 0) return SAGE_OK;
  return launch_e2m1(x, out, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAGE_OK
                                                                                   : SAGE_ERR_CUDA;
}

int sage_debug_export_fp16(const void* workspace, int batch, int heads_q, int heads_kv,
                           int seqlen_q, int seqlen_k, int head_dim, int qk_quant_gran,
                           uint16_t* q16, uint16_t* k16, uint16_t* v16, void* stream) {
  Layout L;
  if (!workspace ||
      !make_layout(false, batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim, qk_quant_gran, &L))
    return SAGE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(workspace);
  const int pq = static_cast<int>(L.planes_q), pk = static_cast<int>(L.planes_kv);
  bool ok = true;
  if (q16) ok &= launch_export_fp16(reinterpret_cast<const __half*>(w + L.off_qc), L.q_rows, L.dp,
                                    head_dim, pq, seqlen_q, q16, st) == cudaSuccess;
  if (k16) ok &= launch_export_fp16(reinterpret_cast<const __half*>(w + L.off_kc), L.k_rows, L.dp,
                                    head_dim, pk, seqlen_k, k16, st) == cudaSuccess;
  if (v16) ok &= launch_export_vt16(reinterpret_cast<const __half*>(w + L.off_vt), L.vt_pitch,
                                    L.dp, head_dim, pk, seqlen_k, v16, st) == cudaSuccess;
  return ok ? SAGE_OK : SAGE_ERR_CUDA;
}

int sage_debug_e4m3(const float* x, uint8_t* out, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!x || !out))) return SAGE_ERR_INVALID_ARG;
  if (n == 0) return SAGE_OK;
  return launch_e4m3(x, out, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAGE_OK
                                                                                   : SAGE_ERR_CUDA;
}

}  // extern "C"
