/*
 * sageattn.h — C ABI of libsageattn.so: SageAttention-style quantized attention forward,
 * O = softmax(Q K^T · sm_scale) V, for one NVIDIA GB300 (sm_103a).
 *
 * The operation (pwwt.cn "SageAttention deployment pitfalls guide"):
 *   §1   Q and K are quantized to INT8 with fine-grained scales and QK^T runs on the
 *        8-bit values; V is quantized to FP8 and P·V runs with FP16/FP32 accumulators;
 *        the output stays FP16/BF16.
 *   §4.1 sageattn(q, k, v, tensor_layout="HND"|"NHD", is_causal, sm_scale=None,
 *        return_lse): inputs FP16 or BF16 on one device with one dtype, last dimension
 *        contiguous; head_dim below 64 is zero-padded to 64, between 64 and 128 to 128,
 *        above 128 is an error; Hq must be a multiple of Hkv (GQA); Nq may differ from Nk.
 *   §4.2 qk_quant_gran (per_warp / per_thread; per_block added), pv_accum_dtype
 *        (fp16 / fp32 / fp16+fp32), smooth_k (subtract K's mean over the sequence),
 *        smooth_v (same for V).
 *   §4 (end) sageattn_varlen: variable-length batches given by cu_seqlens_q / cu_seqlens_k.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device pointers on the current device; the caller
 *     owns every buffer (inputs, outputs, LSE, workspace). The library never allocates or
 *     frees device memory, never synchronises inside sage_attn / sage_attn_varlen, and
 *     enqueues all work on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Arguments are validated on the host before anything is launched: on a non-zero
 *     return nothing was written. Errors found on the device (a bad cu_seqlens, a value
 *     too large for the exact mean, a pipeline wait that timed out) are recorded in the
 *     workspace and read back with sage_read_device_status().
 *   - Strides are in elements. The channel (head_dim) stride is always 1.
 *   - The workspace must be 256-byte aligned, at least sage_attn_workspace_size() bytes,
 *     and must not be shared by calls that may run concurrently.
 *   - Thread safety: calls from several host threads are safe; the only global state is a
 *     per-device cache of the kernels' shared-memory opt-in (and of whether the device is
 *     supported). A cudaDeviceReset clears the opt-in but not the cache: do not reset a
 *     device the library has already launched on.
 */
#ifndef SAGEATTN_H
#define SAGEATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, Nk == 0 with Nq > 0 */
  SAGE_ERR_HEAD_DIM = 2,     /* head_dim < 1 or > 128 */
  SAGE_ERR_DTYPE = 3,        /* dtype not SAGE_F16 / SAGE_BF16 */
  SAGE_ERR_STRIDE = 4,       /* misaligned pointer or a stride that breaks the layout rules */
  SAGE_ERR_GQA = 5,          /* Hq not a multiple of Hkv */
  SAGE_ERR_WORKSPACE = 6,    /* workspace null, misaligned or too small */
  SAGE_ERR_RANGE = 7,        /* (device) |x| >= 2^38 / N: too large for the exact mean */
  SAGE_ERR_UNSUPPORTED = 8,  /* pv_accum_dtype SAGE_ACC_FP16 */
  SAGE_ERR_TIMEOUT = 9,      /* (device) a bounded pipeline wait expired */
  SAGE_ERR_CUDA = 10,        /* a CUDA runtime/driver call failed */
  SAGE_ERR_DEVICE = 11,      /* current device is not compute capability 10.3 */
  SAGE_ERR_SEQLENS = 12      /* (device) cu_seqlens not non-decreasing / out of range */
} sage_status;

enum { SAGE_HND = 0, SAGE_NHD = 1 };                       /* §4.1 tensor_layout */
enum { SAGE_F16 = 0, SAGE_BF16 = 1 };                      /* input/output dtype */
enum { SAGE_PER_BLOCK = 0, SAGE_PER_WARP = 1, SAGE_PER_THREAD = 2 };   /* qk_quant_gran */
enum { SAGE_ACC_FP32 = 0, SAGE_ACC_FP16_FP32 = 1, SAGE_ACC_FP32_FP32 = 2, SAGE_ACC_FP16 = 3 };

/* A 4-d FP16/BF16 device tensor in the order the call's tensor_layout names:
 * HND = [batch, heads, seq, head_dim], NHD = [batch, seq, heads, head_dim].
 * stride[0..2] are the element strides of the first three dimensions; the fourth
 * (channel) stride is 1. `data` points at element [0, 0, 0, 0]. */
typedef struct {
  void* data;
  int64_t stride[3];
} sage_tensor;

/* A packed variable-length FP16/BF16 device tensor [total_tokens, heads, head_dim]
 * with element strides per token and per head; the channel stride is 1. */
typedef struct {
  void* data;
  int64_t stride_token;
  int64_t stride_head;
} sage_packed;

/* Bytes of workspace sage_attn needs for these sizes (0 on invalid sizes). */
size_t sage_attn_workspace_size(int batch, int heads_q, int heads_kv, int seqlen_q,
                                int seqlen_k, int head_dim, int qk_quant_gran);

/* Dense forward (§4.1, §4.2).
 *   q [B, Hq, Nq, d] / [B, Nq, Hq, d]; k, v [B, Hkv, Nk, d] / [B, Nk, Hkv, d] (device,
 *   read only); out: same shape and layout as q (device, written, dtype = input dtype).
 *   lse: device float [B, Hq, Nq] contiguous, natural-log log-sum-exp of the scaled
 *   scores sm_scale·q·k over the allowed keys; written only when return_lse != 0
 *   (may be NULL otherwise).
 *   is_causal: key j is allowed for query i iff j <= i (top-left aligned, as
 *   torch.nn.functional.scaled_dot_product_attention).
 *   sm_scale: scale of the scores; NaN or <= 0 selects 1/sqrt(head_dim).
 *   qk_quant_gran: token groups sharing one INT8 scale — per_block 128 Q rows / 64 K rows,
 *   per_warp 32 / 64, per_thread 1 / 16.
 *   pv_accum_dtype: SAGE_ACC_FP32, SAGE_ACC_FP32_FP32 or SAGE_ACC_FP16_FP32, one
 *   arithmetic on this GPU: P is scaled by 448 before its FP8 rounding and P·V accumulates
 *   in fp32 over every key (§4.2 ranks fp16 accumulation fastest and fp32 most stable, with
 *   fp16+fp32 between them; the tensor cores here accumulate fp16 no faster than fp32, so the
 *   compromise is taken at fp32); SAGE_ACC_FP16 returns SAGE_ERR_UNSUPPORTED.
 *   smooth_k / smooth_v: subtract the per-(batch, head, channel) mean over the sequence.
 *   Nq == 0 or B == 0 is a no-op returning SAGE_OK.
 * Returns a sage_status. */
int sage_attn(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
              const sage_tensor* out, float* lse, int batch, int heads_q, int heads_kv,
              int seqlen_q, int seqlen_k, int head_dim, int dtype, int tensor_layout,
              int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
              int pv_accum_dtype, int smooth_k, int smooth_v, void* workspace,
              size_t workspace_bytes, void* stream);

/* FP16 P·V variant (pwwt.cn "SageAttention deployment pitfalls guide" §5.3–§5.4: the INT8-QK
 * + FP16-PV kernel, the quality fallback with FP8 turned off): as sage_attn, with the same
 * arguments, workspace size and errors, except that V' = V - v̄ is kept in fp16 (no per-channel
 * scale) and P = 2^(t - m) is rounded to fp16 (σ_P = 1); both P·V operands are fp16 on the
 * tensor cores (kind::f16) with fp32 accumulation. pv_accum_dtype: SAGE_ACC_FP32,
 * SAGE_ACC_FP32_FP32 or SAGE_ACC_FP16_FP32 (one arithmetic, as for sage_attn);
 * SAGE_ACC_FP16 returns SAGE_ERR_UNSUPPORTED. |V - v̄| beyond the fp16 range becomes ±inf. */
int sage_attn_qk_int8_pv_fp16(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                              const sage_tensor* out, float* lse, int batch, int heads_q,
                              int heads_kv, int seqlen_q, int seqlen_k, int head_dim, int dtype,
                              int tensor_layout, int is_causal, float sm_scale, int return_lse,
                              int qk_quant_gran, int pv_accum_dtype, int smooth_k, int smooth_v,
                              void* workspace, size_t workspace_bytes, void* stream);

/* FP4 microscaled variant (pwwt.cn "SageAttention deployment pitfalls guide" §5.5: the
 * SageAttention3 kernel for Blackwell, "FP4 microscaling"; the guide names only its API,
 * sageattn3_blackwell(q, k, v, is_causal)): as sage_attn, with the same arguments, workspace
 * size and errors, except for the quantisation:
 *   Q and K' = K - k̄: each token group (qk_quant_gran) is mapped onto [-448, 448] by its
 *   scale g = absmax / 448; every 16 channels of a row share an E4M3 block scale s (the
 *   block's largest mapped magnitude, rounded) and each element is the E2M1 code of
 *   fl32(u · fl32(6 / s)), RNE, saturating at ±6.
 *   V' = V - v̄: each channel is mapped by absmax_c / 448 and blocked over 16 tokens.
 *   P: 448 · 2^(t - m), blocked over 16 keys.
 * Every E2M1 code times its E4M3 block scale is exact in fp16, so both products run on
 * fp16 tensor cores (kind::f16) and give what a block-scaled FP4 product gives. P·V
 * accumulates in fp32; pv_accum_dtype as for sage_attn. Dense problems only. */
int sage_attn_fp4(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                  const sage_tensor* out, float* lse, int batch, int heads_q, int heads_kv,
                  int seqlen_q, int seqlen_k, int head_dim, int dtype, int tensor_layout,
                  int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
                  int pv_accum_dtype, int smooth_k, int smooth_v, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Capacity of the scratch array built into the library for sage_attn_no_alloc. */
#define SAGE_NO_ALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* sage_attn without a caller-supplied workspace and without any device allocation.
 * (The pages have no counterpart; this exists for callers that cannot allocate.)
 * Some callers cannot call cudaMalloc where they run attention: a plugin executing inside a
 * host engine that gives it only its input/output buffers and forbids allocation while it
 * runs, or a latency-critical path that cannot afford an allocation's time or failure. This
 * entry point takes its scratch from a fixed array of SAGE_NO_ALLOC_SCRATCH_BYTES bytes
 * compiled into the library (held by every GPU that loads the library until the process
 * exits); the caller still passes inputs, outputs and the optional LSE buffer.
 *   Arguments, layouts and results are those of sage_attn.
 *   Returns SAGE_ERR_WORKSPACE, before launching anything, when the problem needs more than
 *   SAGE_NO_ALLOC_SCRATCH_BYTES of scratch (sage_attn_workspace_size tells how much).
 *   Arguments are checked first, with sage_attn's rules and error codes.
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current) and caches it for the life of the process; make that first
 *   call before any stream capture. After a cudaDeviceReset the cached address is stale:
 *   do not call this entry point in a process that has reset a device it used.
 *   Every call on a device uses the same array: calls that may overlap on the GPU (other
 *   streams, other host threads) race and must be serialised by the caller. Each call
 *   clears what it needs cleared; nothing an earlier call left in the array is read.
 *   Calls no cudaMalloc, cudaFree or allocating library routine. */
int sage_attn_no_alloc(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                       const sage_tensor* out, float* lse, int batch, int heads_q, int heads_kv,
                       int seqlen_q, int seqlen_k, int head_dim, int dtype, int tensor_layout,
                       int is_causal, float sm_scale, int return_lse, int qk_quant_gran,
                       int pv_accum_dtype, int smooth_k, int smooth_v, void* stream);

/* Bytes of workspace sage_attn_varlen needs (0 on invalid sizes). */
size_t sage_attn_varlen_workspace_size(int batch, int heads_q, int heads_kv, int total_q,
                                       int total_k, int head_dim, int qk_quant_gran);

/* Variable-length forward (§4, sageattn_varlen). Sequence b owns query tokens
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q and key tokens [cu_seqlens_k[b],
 * cu_seqlens_k[b+1]) of k and v; smoothing means, quantisation groups and the causal mask
 * restart per sequence.
 *   q, out: [total_q, Hq, d]; k, v: [total_k, Hkv, d] (device).
 *   cu_seqlens_q, cu_seqlens_k: device int32 [batch + 1], non-decreasing, starting at 0
 *   and ending at total_q / total_k (checked on the device: SAGE_ERR_SEQLENS).
 *   max_seqlen_q / max_seqlen_k: upper bounds of the lengths (checked on the device).
 *   lse: device float [Hq, total_q] when return_lse != 0.
 *   A sequence with no keys but some queries is a device error (SAGE_ERR_SEQLENS).
 * Other arguments as sage_attn. */
int sage_attn_varlen(const sage_packed* q, const sage_packed* k, const sage_packed* v,
                     const sage_packed* out, float* lse, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_k, int batch, int max_seqlen_q,
                     int max_seqlen_k, int total_q, int total_k, int heads_q, int heads_kv,
                     int head_dim, int dtype, int is_causal, float sm_scale, int return_lse,
                     int qk_quant_gran, int pv_accum_dtype, int smooth_k, int smooth_v,
                     void* workspace, size_t workspace_bytes, void* stream);

/* The FP16 P·V variant of sage_attn_varlen (see sage_attn_qk_int8_pv_fp16): same arguments,
 * workspace size and errors; V' and P in fp16 on the tensor cores. */
int sage_attn_varlen_qk_int8_pv_fp16(const sage_packed* q, const sage_packed* k,
                                     const sage_packed* v, const sage_packed* out, float* lse,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int batch, int max_seqlen_q, int max_seqlen_k, int total_q,
                                     int total_k, int heads_q, int heads_kv, int head_dim,
                                     int dtype, int is_causal, float sm_scale, int return_lse,
                                     int qk_quant_gran, int pv_accum_dtype, int smooth_k,
                                     int smooth_v, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* Composition of partial results over disjoint key sets (pwwt.cn "SageAttention deployment
 * pitfalls guide" §4.1: return_lse exists for Ring Attention and similar schemes, which attend
 * to chunks of the keys separately). For every (b, h, n) row:
 *   lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) * out_i
 * computed in fp32 and rounded once to `dtype`.
 *   outs[0..n_parts): device tensors in `tensor_layout` (as sage_attn's out, dtype `dtype`);
 *   lses[0..n_parts): device float [B, H, N] contiguous (as sage_attn writes them);
 *   out: device tensor of the same shape (may alias outs[0]); lse_out: device float
 *   [B, H, N] or NULL. The pointer arrays themselves are host memory.
 * A part whose lse is -inf contributes nothing; a row no part sees gets out = 0 and
 * lse = -inf. 1 <= n_parts <= SAGE_MAX_MERGE_PARTS. Errors: SAGE_ERR_INVALID_ARG (counts,
 * null pointers, layout), SAGE_ERR_DTYPE, SAGE_ERR_HEAD_DIM, SAGE_ERR_STRIDE (pointer not
 * 2-byte aligned, negative stride), SAGE_ERR_CUDA. Nothing is launched for an empty problem. */
#define SAGE_MAX_MERGE_PARTS 16
int sage_merge_partials(const sage_tensor* outs, const float* const* lses, int n_parts,
                        const sage_tensor* out, float* lse_out, int batch, int heads,
                        int seqlen, int head_dim, int dtype, int tensor_layout, void* stream);

/* Human-readable name of a sage_status. Never NULL. */
const char* sage_status_string(int status);

/* Name and description of the CUDA error behind the calling thread's most recent
 * SAGE_ERR_CUDA ("no error" if there was none). Never NULL. */
const char* sage_last_cuda_error(void);

/* Synchronises `stream`, then returns the status the device recorded in `workspace`
 * during the last call that used it (SAGE_OK if none), or SAGE_ERR_CUDA. */
int sage_read_device_status(const void* workspace, void* stream);

/* 1 if the current CUDA device is compute capability 10.3 (GB300), else 0. */
int sage_device_supported(void);

/* Stage timing (off by default). While enabled, every sage_attn / sage_attn_varlen call
 * records CUDA events on its stream around its three stages (statistics, quantisation,
 * attention kernel); up to 8192 calls are kept. sage_profile_read synchronises those events
 * and writes the summed milliseconds per stage to stage_ms[0..2] and the number of calls to
 * *calls; it also clears the record. Enabling allocates CUDA events (no device memory).
 * Returns a sage_status. */
int sage_profile_enable(int on);
int sage_profile_read(double* stage_ms, int* calls);

/* ---- Test exports. They run the same kernels as the entry points above. ---- */

/* Copies the quantised state that the last sage_attn call with these sizes left in
 * `workspace` into canonical host-layout device buffers (all device, caller-owned):
 *   q8 int8 [B, Hq, Nq, d], sq float [B, Hq, ceil(Nq / Gq)],
 *   k8 int8 [B, Hkv, Nk, d], sk float [B, Hkv, ceil(Nk / Gk)],
 *   kmean, vmean, vscale float [B, Hkv, d], v8 uint8 E4M3 [B, Hkv, Nk, d].
 * Any output pointer may be NULL to skip it. */
int sage_debug_export_quant(const void* workspace, int batch, int heads_q, int heads_kv,
                            int seqlen_q, int seqlen_k, int head_dim, int qk_quant_gran,
                            int8_t* q8, float* sq, int8_t* k8, float* sk, float* kmean,
                            float* vmean, float* vscale, uint8_t* v8, void* stream);

/* sage_attn that additionally writes the integer scores S = Q8 · K8^T, exactly as the
 * attention kernel reads them from tensor memory, to `scores` (device int32
 * [B, Hq, Nq, Nk]; entries the causal mask skips are left untouched). */
int sage_attn_debug_scores(const sage_tensor* q, const sage_tensor* k, const sage_tensor* v,
                           const sage_tensor* out, float* lse, int batch, int heads_q,
                           int heads_kv, int seqlen_q, int seqlen_k, int head_dim, int dtype,
                           int tensor_layout, int is_causal, float sm_scale, int return_lse,
                           int qk_quant_gran, int pv_accum_dtype, int smooth_k, int smooth_v,
                           void* workspace, size_t workspace_bytes, int32_t* scores,
                           void* stream);

/* Test hook: while `on` is non-zero, the attention kernel's producer issues no K/V tile
 * loads, so the consumers' bounded waits expire (about 2 s) and the device status becomes
 * SAGE_ERR_TIMEOUT; the kernel still exits cleanly and the context stays usable. Process-wide;
 * not for concurrent use. Returns SAGE_OK. */
int sage_debug_stall_attention(int on);

/* Which implementation dense sage_attn calls use. The main pipeline is the statistics,
 * finalisation, quantisation and tcgen05 attention kernels (four launches); the short-sequence
 * kernel (pnsm.cn §10: below about 1K tokens fixed costs dominate) takes problems with at most
 * 256 keys and 1024 queries in one launch, doing the statistics, quantisation and attention per
 * CTA of 128 query rows with the same arithmetic and results within the same tolerances.
 *   0 (default): the short-sequence kernel for such problems at head_dim <= 64 on a stream that
 *      is not capturing a CUDA graph, the main pipeline otherwise (measured faster in each
 *      case: 28 us against 37 per direct call at 256 keys; 22 us against 27 replayed);
 *   1: always the main pipeline;
 *   2: the short-sequence kernel whenever the problem fits it.
 * The FP16 P·V and FP4 variants and calls with the score dump, trace or stall hooks always take
 * the main pipeline. Process-wide; not for concurrent use. Returns SAGE_OK, or
 * SAGE_ERR_INVALID_ARG for another value. */
int sage_debug_select_path(int path);

/* Pipeline trace hook: while `clocks` (device, 4*64*8 int64, caller-owned) is non-NULL, dense
 * calls record clock64() of the first CTA's pipeline events there: [role][tile][event] with
 * role 0/1 = softmax of query tile A/B (events: scores ready, scores loaded, max done,
 * exponentials done, P buffer free, P written, O rescaled; event 7 of the last tile: output
 * written), role 2 = MMA issue (per tile x:
 * 4x+0 P ready, 4x+1 QK^T issued, 4x+2 O ready, 4x+3 P.V issued), role 3 = TMA (K, V
 * issued), for the first 64 KV tiles. NULL turns it off. Process-wide. Returns SAGE_OK.
 * The events are recorded by a separate test build of the E4M3 P·V attention kernel (the
 * production build carries no trace points, so its timing differs); calls of the FP16 P·V
 * and FP4 variants record nothing. */
int sage_debug_trace_attention(long long* clocks);

/* Converts n floats (device) to FP8 E4M3 (device bytes) with the round-to-nearest-even,
 * saturating conversion the kernels use for V and P. */
int sage_debug_e4m3(const float* x, uint8_t* out, int64_t n, void* stream);

/* Converts n floats (device) to FP4 E2M1 codes (device bytes, low 4 bits) with the
 * round-to-nearest-even conversion saturating at ±6 that the FP4 variant uses. */
int sage_debug_e2m1(const float* x, uint8_t* out, int64_t n, void* stream);

/* Copies the fp16 operands the attention kernel consumed after a dense call of the FP16 P·V
 * or FP4 variant into canonical layouts (device buffers of fp16 bit patterns):
 *   q16 [B, Hq, Nq, d] and k16 [B, Hkv, Nk, d] (the FP4 carriers; INT8 codes as fp16 after
 *   the other dense calls), v16 [B, Hkv, Nk, d] (V' in fp16, or the FP4 carriers of V).
 * Any output pointer may be NULL to skip it. */
int sage_debug_export_fp16(const void* workspace, int batch, int heads_q, int heads_kv,
                           int seqlen_q, int seqlen_k, int head_dim, int qk_quant_gran,
                           uint16_t* q16, uint16_t* k16, uint16_t* v16, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SAGEATTN_H */
