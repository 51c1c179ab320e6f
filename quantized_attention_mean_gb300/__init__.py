"""SageAttention-style quantized attention forward for one GB300 (sm_103a).

Thin Python binding over libsageattn.so (include/sageattn.h). PyTorch only supplies device
memory and streams; every step of the computation runs in the library's CUDA kernels.

    out = sage_attn(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None,
                    return_lse=False, qk_quant_gran="per_warp", pv_accum_dtype="fp32",
                    smooth_k=True, smooth_v=False)

mirrors the ``sageattn`` API (pwwt.cn "SageAttention deployment pitfalls guide" §4.1, §4.2);
``sage_attn_varlen`` mirrors ``sageattn_varlen``; ``merge_partials`` combines results over
disjoint key chunks through their log-sum-exp (ring / context-parallel composition).
"""

import ctypes
import math

import torch

from . import _lib
from ._lib import SagePacked, SageTensor

GRAN = {"per_block": 0, "per_warp": 1, "per_thread": 2}
ACC = {"fp32": 0, "fp16+fp32": 1, "fp32+fp32": 2, "fp16": 3}
LAYOUT = {"HND": 0, "NHD": 1}
DTYPE = {torch.float16: 0, torch.bfloat16: 1}


class SageError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        lib = _lib.load()
        msg = lib.sage_status_string(status).decode()
        if status == 10:  # SAGE_ERR_CUDA: name the failing call
            msg += " [" + lib.sage_last_cuda_error().decode() + "]"
        super().__init__(f"{what}: {msg}" if what else msg)


def _check(status, what):
    if status != 0:
        raise SageError(status, what)


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _tensor(t):
    st = t.stride()
    if st[3] != 1:
        raise ValueError("the last dimension must be contiguous")
    return SageTensor(t.data_ptr(), (ctypes.c_int64 * 3)(st[0], st[1], st[2]))


def _packed(t):
    st = t.stride()
    if st[2] != 1:
        raise ValueError("the last dimension must be contiguous")
    return SagePacked(t.data_ptr(), st[0], st[1])


def workspace_bytes(batch, heads_q, heads_kv, seqlen_q, seqlen_k, head_dim, qk_quant_gran="per_warp"):
    return _lib.load().sage_attn_workspace_size(batch, heads_q, heads_kv, seqlen_q, seqlen_k,
                                                head_dim, GRAN[qk_quant_gran])


def varlen_workspace_bytes(batch, heads_q, heads_kv, total_q, total_k, head_dim,
                           qk_quant_gran="per_warp"):
    return _lib.load().sage_attn_varlen_workspace_size(batch, heads_q, heads_kv, total_q, total_k,
                                                       head_dim, GRAN[qk_quant_gran])


def alloc_workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _check_workspace(workspace, device):
    if workspace is not None and (workspace.dtype != torch.uint8 or workspace.device != device
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")


def _check_dense_args(q, k, v, tensor_layout, out, lse, return_lse, workspace):
    """Shapes, dtypes and devices of a dense call. The C ABI sees only pointers and strides,
    so a v smaller than k, or an out / lse smaller than q's, would be read or written past its
    end: such arguments are rejected here, before anything is launched."""
    if tensor_layout not in LAYOUT:
        raise ValueError("tensor_layout must be 'HND' or 'NHD'")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float16 or bfloat16")
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("v must have k's shape")
    B, Hq, _, Nq, _, d = _dims(q, k, tensor_layout)
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k must have q's batch size and head_dim")
    if out is not None and (tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype
                            or out.device != q.device):
        raise ValueError("out must have q's shape, dtype and device")
    if return_lse and lse is not None and (tuple(lse.shape) != (B, Hq, Nq) or lse.dtype != torch.float32
                                           or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, Hq, Nq] tensor on q's device")
    if not (q.is_cuda and k.device == q.device and v.device == q.device):
        raise ValueError("q, k, v must be on one CUDA device")
    _check_workspace(workspace, q.device)


def _dims(q, k, layout):
    if layout == "HND":
        return q.shape[0], q.shape[1], k.shape[1], q.shape[2], k.shape[2], q.shape[3]
    return q.shape[0], q.shape[2], k.shape[2], q.shape[1], k.shape[1], q.shape[3]


def sage_attn(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None, return_lse=False,
              qk_quant_gran="per_warp", pv_accum_dtype="fp32", smooth_k=True, smooth_v=False,
              out=None, lse=None, workspace=None, stream=None, _debug_scores=None, _pv16=False,
              _fp4=False):
    """Quantized attention forward. q: [B, Hq, Nq, d] (HND) or [B, Nq, Hq, d] (NHD);
    k, v: [B, Hkv, Nk, d] / [B, Nk, Hkv, d]; fp16 or bf16 on one CUDA device.
    Returns out (same shape/layout/dtype as q), plus lse [B, Hq, Nq] fp32 if return_lse."""
    lib = _lib.load()
    _check_dense_args(q, k, v, tensor_layout, out, lse, return_lse, workspace)
    B, Hq, Hkv, Nq, Nk, d = _dims(q, k, tensor_layout)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    need = lib.sage_attn_workspace_size(B, Hq, Hkv, Nq, Nk, d, GRAN[qk_quant_gran])
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    scale = float("nan") if sm_scale is None else float(sm_scale)
    args = [ctypes.byref(_tensor(q)), ctypes.byref(_tensor(k)), ctypes.byref(_tensor(v)),
            ctypes.byref(_tensor(out)), ctypes.c_void_p(lse.data_ptr() if return_lse else 0),
            B, Hq, Hkv, Nq, Nk, d, DTYPE[q.dtype], LAYOUT[tensor_layout], int(bool(is_causal)),
            scale, int(bool(return_lse)), GRAN[qk_quant_gran], ACC[pv_accum_dtype],
            int(bool(smooth_k)), int(bool(smooth_v)), ctypes.c_void_p(workspace.data_ptr()),
            workspace.numel()]
    with torch.cuda.device(q.device):
        if _fp4:
            st = lib.sage_attn_fp4(*args, _stream_ptr(stream))
        elif _pv16:
            st = lib.sage_attn_qk_int8_pv_fp16(*args, _stream_ptr(stream))
        elif _debug_scores is None:
            st = lib.sage_attn(*args, _stream_ptr(stream))
        else:
            st = lib.sage_attn_debug_scores(*args, ctypes.c_void_p(_debug_scores.data_ptr()),
                                            _stream_ptr(stream))
    _check(st, "sage_attn")
    return (out, lse) if return_lse else out


def sage_attn_qk_int8_pv_fp16(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None,
                              return_lse=False, qk_quant_gran="per_warp", pv_accum_dtype="fp32",
                              smooth_k=True, smooth_v=False, out=None, lse=None, workspace=None,
                              stream=None):
    """The FP16 P·V variant (INT8 Q/K; P and V' in fp16 on the tensor cores), mirroring the
    pages' ``sageattn_qk_int8_pv_fp16_cuda`` quality fallback. Arguments and results as
    ``sage_attn``."""
    return sage_attn(q, k, v, tensor_layout=tensor_layout, is_causal=is_causal, sm_scale=sm_scale,
                     return_lse=return_lse, qk_quant_gran=qk_quant_gran,
                     pv_accum_dtype=pv_accum_dtype, smooth_k=smooth_k, smooth_v=smooth_v, out=out,
                     lse=lse, workspace=workspace, stream=stream, _pv16=True)


def sage_attn_fp4(q, k, v, tensor_layout="HND", is_causal=False, sm_scale=None, return_lse=False,
                  qk_quant_gran="per_warp", pv_accum_dtype="fp32", smooth_k=True, smooth_v=False,
                  out=None, lse=None, workspace=None, stream=None):
    """The FP4 microscaled variant (E2M1 codes with E4M3 scales per 16 elements for Q, K, P
    and V), standing for the pages' ``sageattn3_blackwell``. Arguments and results as
    ``sage_attn``."""
    return sage_attn(q, k, v, tensor_layout=tensor_layout, is_causal=is_causal, sm_scale=sm_scale,
                     return_lse=return_lse, qk_quant_gran=qk_quant_gran,
                     pv_accum_dtype=pv_accum_dtype, smooth_k=smooth_k, smooth_v=smooth_v, out=out,
                     lse=lse, workspace=workspace, stream=stream, _fp4=True)


def sage_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                     is_causal=False, sm_scale=None, return_lse=False, qk_quant_gran="per_warp",
                     pv_accum_dtype="fp32", smooth_k=True, smooth_v=False, out=None, lse=None,
                     workspace=None, stream=None, pv="fp8"):
    """Variable-length forward: q [Tq, Hq, d], k/v [Tk, Hkv, d], cu_seqlens int32 [B+1] on the
    device. Returns out [Tq, Hq, d] (+ lse [Hq, Tq] fp32 if return_lse). pv="fp16" selects the
    FP16 P·V variant."""
    lib = _lib.load()
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be packed 3-D [tokens, heads, head_dim] tensors")
    if q.dtype not in DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype, float16 or bfloat16")
    if tuple(v.shape) != tuple(k.shape) or k.shape[2] != q.shape[2]:
        raise ValueError("v must have k's shape, and k q's head_dim")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if (cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape != cu_seqlens_k.shape or cu_seqlens_q.numel() < 1
            or not cu_seqlens_q.is_contiguous() or not cu_seqlens_k.is_contiguous()):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be contiguous 1-D [batch + 1] tensors")
    if out is not None and (tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype
                            or out.device != q.device):
        raise ValueError("out must have q's shape, dtype and device")
    if return_lse and lse is not None and (tuple(lse.shape) != (q.shape[1], q.shape[0])
                                           or lse.dtype != torch.float32 or not lse.is_contiguous()
                                           or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [Hq, total_q] tensor on q's device")
    if not (q.is_cuda and k.device == q.device and v.device == q.device
            and cu_seqlens_q.device == q.device and cu_seqlens_k.device == q.device):
        raise ValueError("q, k, v and cu_seqlens must be on one CUDA device")
    _check_workspace(workspace, q.device)
    Tq, Hq, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    need = lib.sage_attn_varlen_workspace_size(B, Hq, Hkv, Tq, Tk, d, GRAN[qk_quant_gran])
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    scale = float("nan") if sm_scale is None else float(sm_scale)
    with torch.cuda.device(q.device):
        if pv not in ("fp8", "fp16"):
            raise ValueError("pv must be 'fp8' or 'fp16'")
        entry = lib.sage_attn_varlen_qk_int8_pv_fp16 if pv == "fp16" else lib.sage_attn_varlen
        st = entry(
            ctypes.byref(_packed(q)), ctypes.byref(_packed(k)), ctypes.byref(_packed(v)),
            ctypes.byref(_packed(out)), ctypes.c_void_p(lse.data_ptr() if return_lse else 0),
            ctypes.c_void_p(cu_seqlens_q.data_ptr()), ctypes.c_void_p(cu_seqlens_k.data_ptr()),
            B, int(max_seqlen_q), int(max_seqlen_k), Tq, Tk, Hq, Hkv, d, DTYPE[q.dtype],
            int(bool(is_causal)), scale, int(bool(return_lse)), GRAN[qk_quant_gran],
            ACC[pv_accum_dtype], int(bool(smooth_k)), int(bool(smooth_v)),
            ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    _check(st, "sage_attn_varlen")
    return (out, lse) if return_lse else out


def merge_partials(outs, lses, tensor_layout="HND", out=None, lse=None, stream=None):
    """Combines attention results computed over disjoint key sets (each from ``sage_attn``
    with ``return_lse=True``): lse = ln sum_i exp(lse_i), out = sum_i exp(lse_i - lse) out_i.
    outs: tensors of one shape/layout/dtype ([B, H, N, d] HND or [B, N, H, d] NHD); lses:
    fp32 [B, H, N]. Returns (out, lse)."""
    lib = _lib.load()
    if len(outs) != len(lses) or not outs:
        raise ValueError("one lse per partial output, at least one part")
    o0 = outs[0]
    if o0.dtype not in DTYPE or any(o.dtype != o0.dtype or o.shape != o0.shape for o in outs):
        raise TypeError("partial outputs must share one shape and a float16/bfloat16 dtype")
    if tensor_layout == "HND":
        B, H, N, d = o0.shape
    else:
        B, N, H, d = o0.shape
    for l in lses:
        if l.dtype != torch.float32 or tuple(l.shape) != (B, H, N) or not l.is_contiguous():
            raise ValueError("each lse must be a contiguous float32 [B, H, N] tensor")
    if out is not None and (tuple(out.shape) != tuple(o0.shape) or out.dtype != o0.dtype):
        raise ValueError("out must have the partial outputs' shape and dtype")
    if lse is not None and (tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    devs = {t.device for t in list(outs) + list(lses) + [x for x in (out, lse) if x is not None]}
    if len(devs) != 1 or not o0.is_cuda:
        raise ValueError("all tensors must be on one CUDA device")
    if out is None:
        out = torch.empty_like(o0)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o0.device)
    views = (SageTensor * len(outs))(*[_tensor(o) for o in outs])
    ptrs = (ctypes.c_void_p * len(lses))(*[l.data_ptr() for l in lses])
    with torch.cuda.device(o0.device):
        st = lib.sage_merge_partials(ctypes.cast(views, ctypes.c_void_p), ctypes.cast(ptrs, ctypes.c_void_p),
                                     len(outs), ctypes.byref(_tensor(out)),
                                     ctypes.c_void_p(lse.data_ptr()), B, H, N, d, DTYPE[o0.dtype],
                                     LAYOUT[tensor_layout], _stream_ptr(stream))
    _check(st, "sage_merge_partials")
    return out, lse


def scaled_dot_product_attention(query, key, value, attn_mask=None, dropout_p=0.0,
                                 is_causal=False, scale=None, enable_gqa=False, **sage_kwargs):
    """Stand-in for ``torch.nn.functional.scaled_dot_product_attention`` on the quantized path
    (the pages present the method as a replacement for that call; pwwt.cn "SageAttention
    deployment pitfalls guide" §4.1, §5.1: a one-line replacement of that function; masks
    other than causal are not supported).

    query [B, H, L, d] or [H, L, d]; key / value [B, Hkv, S, d] or [Hkv, S, d] (HND), fp16 or
    bf16, head_dim <= 128. ``is_causal`` masks key j for query i when j > i (top-left, as
    torch). ``scale`` defaults to 1/sqrt(d). Key/value heads may divide the query heads
    (grouped-query attention) whatever ``enable_gqa`` says. Arbitrary masks and dropout are
    not supported by the method and raise NotImplementedError. Extra keyword arguments go to
    ``sage_attn`` (qk_quant_gran, pv_accum_dtype, smooth_k, smooth_v)."""
    if attn_mask is not None:
        raise NotImplementedError("attn_mask: the quantized kernel supports only causal or no masking")
    if dropout_p != 0.0:
        raise NotImplementedError("dropout_p must be 0")
    if query.dim() not in (3, 4) or key.dim() != query.dim() or value.dim() != query.dim():
        raise ValueError("expected [B, H, N, d] or [H, N, d] tensors")
    squeeze = query.dim() == 3
    if squeeze:
        query, key, value = query.unsqueeze(0), key.unsqueeze(0), value.unsqueeze(0)
    if key.shape[1] == 0 or query.shape[1] % key.shape[1] != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    q, k, v = (t if t.stride(-1) == 1 else t.contiguous() for t in (query, key, value))
    out = sage_attn(q, k, v, tensor_layout="HND", is_causal=is_causal, sm_scale=scale, **sage_kwargs)
    return out.squeeze(0) if squeeze else out


def read_device_status(workspace, stream=None):
    return _lib.load().sage_read_device_status(ctypes.c_void_p(workspace.data_ptr()), _stream_ptr(stream))


def export_quant(workspace, B, Hq, Hkv, Nq, Nk, d, qk_quant_gran, stream=None):
    """Copies the quantised tensors a previous dense sage_attn left in `workspace`."""
    lib = _lib.load()
    g = GRAN[qk_quant_gran]
    gq, gk = {0: (128, 64), 1: (32, 64), 2: (1, 16)}[g]
    dev = workspace.device
    res = dict(
        q8=torch.empty((B, Hq, Nq, d), dtype=torch.int8, device=dev),
        sq=torch.empty((B, Hq, -(-Nq // gq)), dtype=torch.float32, device=dev),
        k8=torch.empty((B, Hkv, Nk, d), dtype=torch.int8, device=dev),
        sk=torch.empty((B, Hkv, -(-Nk // gk)), dtype=torch.float32, device=dev),
        kmean=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev),
        vmean=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev),
        vscale=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev),
        v8=torch.empty((B, Hkv, Nk, d), dtype=torch.uint8, device=dev),
    )
    order = ["q8", "sq", "k8", "sk", "kmean", "vmean", "vscale", "v8"]
    st = lib.sage_debug_export_quant(ctypes.c_void_p(workspace.data_ptr()), B, Hq, Hkv, Nq, Nk, d, g,
                                     *[ctypes.c_void_p(res[n].data_ptr()) for n in order],
                                     _stream_ptr(stream))
    _check(st, "sage_debug_export_quant")
    return res


def export_fp16(workspace, B, Hq, Hkv, Nq, Nk, d, qk_quant_gran, stream=None):
    """Copies the fp16 operands (Q and K codes or FP4 carriers, V' in fp16 or its FP4
    carriers) a previous dense call of the FP16 P·V or FP4 variant left in `workspace`, as
    float16 tensors [B, H, N, d]."""
    lib = _lib.load()
    g = GRAN[qk_quant_gran]
    dev = workspace.device
    res = dict(q16=torch.empty((B, Hq, Nq, d), dtype=torch.float16, device=dev),
               k16=torch.empty((B, Hkv, Nk, d), dtype=torch.float16, device=dev),
               v16=torch.empty((B, Hkv, Nk, d), dtype=torch.float16, device=dev))
    st = lib.sage_debug_export_fp16(ctypes.c_void_p(workspace.data_ptr()), B, Hq, Hkv, Nq, Nk, d, g,
                                    *[ctypes.c_void_p(res[n].data_ptr()) for n in ("q16", "k16", "v16")],
                                    _stream_ptr(stream))
    _check(st, "sage_debug_export_fp16")
    return res


def e2m1(x, stream=None):
    """FP4 E2M1 conversion with the kernels' rounding (test hook): float32 CUDA -> uint8 codes."""
    lib = _lib.load()
    x = x.contiguous()
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib.sage_debug_e2m1(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                               x.numel(), _stream_ptr(stream)), "sage_debug_e2m1")
    return out


def e4m3(x, stream=None):
    """FP8 E4M3 conversion with the kernels' rounding (test hook): float32 CUDA -> uint8."""
    lib = _lib.load()
    x = x.contiguous()
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib.sage_debug_e4m3(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                               x.numel(), _stream_ptr(stream)), "sage_debug_e4m3")
    return out


def select_path(path="auto"):
    """Which implementation dense calls use: "auto" (the one-launch short-sequence kernel for
    head_dim <= 64 problems with at most 256 keys and 1024 queries on a stream that is not
    capturing a CUDA graph, the four-launch main pipeline otherwise), "main" (always the main
    pipeline) or "short" (the short-sequence kernel whenever the problem fits it). Process-wide."""
    _check(_lib.load().sage_debug_select_path({"auto": 0, "main": 1, "short": 2}[path]),
           "sage_debug_select_path")


def profile_enable(on=True):
    _check(_lib.load().sage_profile_enable(int(bool(on))), "sage_profile_enable")


def profile_read():
    """Summed ms per stage [stats, quant, attention] of the calls since enable / last read."""
    ms = (ctypes.c_double * 3)()
    n = ctypes.c_int(0)
    _check(_lib.load().sage_profile_read(ms, ctypes.byref(n)), "sage_profile_read")
    return list(ms), n.value


def default_sm_scale(head_dim):
    return 1.0 / math.sqrt(head_dim)


__all__ = ["sage_attn", "sage_attn_varlen", "sage_attn_fp4", "SageError", "workspace_bytes",
           "varlen_workspace_bytes", "alloc_workspace", "read_device_status", "export_quant",
           "export_fp16", "e4m3", "e2m1",
           "profile_enable", "profile_read"]
