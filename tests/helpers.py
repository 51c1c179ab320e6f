"""Shared test helpers: run the CUDA path and the oracle on the same seeded inputs."""

import numpy as np
import torch

from quantized_attention_mean_gb300.workloads import ACC, GRAN, Workload, dense_inputs, to_hnd_f32

TOL_MAX_ABS = 2e-2      # O vs the oracle's quantised emulation (max-abs)
TOL_COS = 0.9995        # O vs the oracle's quantised emulation (cosine)
TOL_COS_FP64 = 0.99     # O vs float64 unquantised attention (cosine)
TOL_LSE = 2e-2          # LSE vs the oracle (absolute)
# O and LSE vs the oracle's online form (p_max="running"), which quantises P~ the way the
# kernel does. What separates the two is ex2.approx vs exp and fp32 sums; where that tips
# one P~ across an E4M3 rounding boundary, a row that sees only a few keys moves by up to a
# few percent of a V value, so the element bound stays at half the bound above while almost
# every element must agree to 1e-3 (beyond the output's own rounding), and cosine and LSE are
# tight.
TOL_ONLINE_MAX_ABS = 1e-2
TOL_ONLINE_ELEM = 1e-3
TOL_ONLINE_ELEM_FRAC = 1e-3
TOL_ONLINE_COS = 0.99999
TOL_ONLINE_LSE = 1e-4


def out_ulp(x, dtype):
    """One unit in the last place of the output format at |x| (fp16: 11-bit, bf16: 8-bit
    significand)."""
    sig, min_exp = (11, -14) if dtype == "fp16" else (8, -126)
    _, e = np.frexp(np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** min_exp))
    return np.ldexp(1.0, e - sig)


def rounding_excess(o_gpu, o_ref, dtype):
    """|o_gpu - o_ref| minus half an ulp of o_gpu, elementwise. o_gpu is the kernel's fp32
    result rounded once (to nearest) to the output format, which moves it by at most half an
    ulp of the rounded value; what is left bounds the error of the kernel's unrounded result
    against the oracle's exact (float64) value."""
    o_gpu = np.asarray(o_gpu, np.float64)
    return np.abs(o_gpu - o_ref) - 0.5 * out_ulp(o_gpu, dtype)


def max_abs_excess(o_gpu, o_ref, dtype):
    """The largest output error beyond the output format's own final rounding."""
    return float(np.max(rounding_excess(o_gpu, o_ref, dtype)))


def excess_fraction(o_gpu, o_ref, dtype, thr):
    """Fraction of elements whose error beyond the final rounding exceeds thr."""
    return float(np.mean(rounding_excess(o_gpu, o_ref, dtype) > thr))


def assert_online_parity(o_gpu, o_ref, dtype, lse=None, lse_ref=None):
    """The output against the oracle's online form (see the TOL_ONLINE_* bounds)."""
    assert max_abs_excess(o_gpu, o_ref, dtype) <= TOL_ONLINE_MAX_ABS
    assert excess_fraction(o_gpu, o_ref, dtype, TOL_ONLINE_ELEM) <= TOL_ONLINE_ELEM_FRAC
    assert cosine(o_gpu, o_ref) >= TOL_ONLINE_COS
    if lse is not None:
        assert np.abs(np.asarray(lse) - lse_ref).max() <= TOL_ONLINE_LSE


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def oracle_kw(w: Workload, sm_scale=None):
    return dict(is_causal=w.is_causal, sm_scale=sm_scale, gran=GRAN[w.gran], accum=ACC[w.accum],
                smooth_k=w.smooth_k, smooth_v=w.smooth_v)


def gpu_kw(w: Workload):
    return dict(tensor_layout=w.layout, is_causal=w.is_causal, return_lse=w.return_lse,
                qk_quant_gran=w.gran, pv_accum_dtype=w.accum, smooth_k=w.smooth_k,
                smooth_v=w.smooth_v)


def short_eligible(w: Workload):
    """Whether the one-launch short-sequence kernel can take this dense problem."""
    return w.Nk <= 256 and w.Nq <= 1024 and w.extra.get("pv", "fp8") == "fp8"


def run_gpu_dense(w: Workload, q, k, v, sm_scale=None, debug_scores=False, path="auto"):
    """One sage_attn call. path: "auto" / "main" (the main pipeline) or "short" (the one-launch
    short-sequence kernel; the problem must be short_eligible and no score dump requested)."""
    import quantized_attention_mean_gb300 as qa
    assert path != "short" or (short_eligible(w) and not debug_scores)
    qa.select_path(path)
    try:
        return _run_gpu_dense(w, q, k, v, sm_scale, debug_scores)
    finally:
        qa.select_path("auto")


def _run_gpu_dense(w, q, k, v, sm_scale, debug_scores):
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    B, Hq, Hkv, Nq, Nk, d = w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d
    ws = qa.alloc_workspace(qa.workspace_bytes(B, Hq, Hkv, Nq, Nk, d, w.gran), dev)
    scores = None
    if debug_scores:
        scores = torch.full((B, Hq, Nq, Nk), -2**31, dtype=torch.int32, device=dev)
    res = qa.sage_attn(qd, kd, vd, sm_scale=sm_scale, workspace=ws, _debug_scores=scores, **gpu_kw(w))
    out, lse = res if w.return_lse else (res, None)
    torch.cuda.synchronize()
    status = qa.read_device_status(ws)
    return dict(out=out, lse=lse, ws=ws, scores=scores, status=status)


def out_to_hnd(out, layout):
    o = out.float().cpu()
    return (o.transpose(1, 2) if layout == "NHD" else o).numpy()
