"""Stage 3 of the method and the whole forward pass (test oracle).

pwwt.cn "SageAttention deployment pitfalls guide":
  §1   the product QK^T runs on 8-bit integers, P·V on FP8 with FP16/FP32 accumulators,
       the output stays FP16/BF16;
  §4.1 sageattn(q, k, v, tensor_layout, is_causal, sm_scale=None -> 1/sqrt(head_dim),
       return_lse); head_dim padding rule; GQA (Hq divisible by Hkv); Nq may differ
       from Nk;
  §4.2 pv_accum_dtype in {fp16, fp32, fp16+fp32}: all-fp16 fastest but may be unstable,
       fp32 the most stable, fp16+fp32 a compromise between the two;
  §4 (end) sageattn_varlen with cu_seqlens_q / cu_seqlens_k.

The steps, in the order the method applies them, per (batch, query head):
  1. k̄, v̄ = fixed-point means over the sequence (smooth_k / smooth_v; 0 when off)
  2. K' = K - k̄, V' = V - v̄ (float32)
  3. Q, K' -> INT8 per token group; V' -> E4M3 per channel
  4. S = Q8 · K8^T, exact integers
  5. t = S · s_q · s_k · sm_scale, causal mask (key j allowed iff j <= i), in float64
  6. m = row max of t (final max), p = exp(t - m), l = sum p
  7. P~ = e4m3(p · σ_P), σ_P = 448 (the largest E4M3 magnitude)
  8. acc = P~ · V~ as a float64 sum
  9. O = acc · s_v / (σ_P · l) + v̄, rounded once to the output dtype
 10. LSE = m + ln l + sm_scale · (q · k̄)   (natural log; undoes the smooth_k shift)
Steps 5-10 use library matmuls on exact integer or float64 operands only.

Accumulation modes (§4.2): the guide ranks fp16 accumulation as the fastest and fp32 as the
most stable, with fp16+fp32 as the compromise; it gives no other arithmetic for them. On the
tensor cores this library targets an fp16 accumulator is not faster than an fp32 one, so the
compromise costs nothing to resolve in fp32's favour: "fp16+fp32", "fp32+fp32" and "fp32" are
one arithmetic here (σ_P = 448, one sum over every key), and pure "fp16" is not supported.

Online form (p_max="running"): the pages' kernel is flash-style (pnsm.cn §2: tiles of keys
with an online softmax), so P~ can also be read as quantised against the running max of the
keys seen so far. Steps 6-8 then walk the keys in tiles of `key_tile` keys (default 128;
the width is the kernel's choice, so it is a parameter here): per tile, m_new = max(m, tile
max), α = exp(m - m_new) (0 while m = -inf), p = exp(t - m_new), P~ = e4m3(p · σ_P) (fp16 for
the FP16 P·V variant), acc = α · acc + P~ · V~, l = α · l + sum p. Steps 9 and 10 are
unchanged. With one tile, or when every row's maximum lies in its first tile, the two forms
give the same P~.

FP16 P·V variant (pv="fp16"; the guide's §5.3 / §5.4 INT8-QK + FP16-PV kernel, its quality
fallback with FP8 turned off): step 3 keeps V' as fp16 (RNE) instead of E4M3 with a scale,
step 7 rounds P to fp16 with σ_P = 1, and step 9 has no V scale. Steps 4-6, 8 and 10 are
unchanged.

FP4 microscaled variant (pv="fp4"; the guide's §5.5 SageAttention3, "FP4 microscaling", read
as in oracle/fp4.py): step 3 quantises Q and K' to two-level FP4 (first-level scales g_q, g_k
per token group, E4M3 block scales per 16 channels) and V' likewise (g_v per channel, blocks of
16 tokens); each code enters the products as its carrier c · s_b ≈ 6 u. Step 4 multiplies the
carriers (S ≈ 36 · q·k / (g_q g_k)), so step 5 scales by g_q g_k / 36; step 7 quantises
y = fl32(448 p) in blocks of 16 keys (P's carrier ≈ 6 · 448 p: σ_P = 2688); step 9 scales by
g_v / 6. Steps 6, 8 and 10 are unchanged.
"""

import numpy as np

from .fp4 import fp4_channel_quant, fp4_group_quant, fp4_p
from .fp8 import e4m3_decode, e4m3_encode
from .quant import (GRAN_PER_BLOCK, GRAN_PER_THREAD, GRAN_PER_WARP, K_GROUP, Q_GROUP,
                    fixed_point_mean, fp8_channel_quant, int8_group_quant, smooth)

ACC_FP32, ACC_FP16_FP32, ACC_FP32_FP32, ACC_FP16 = 0, 1, 2, 3
KEY_TILE = 128  # default keys per tile of the online form

__all__ = [
    "ACC_FP32", "ACC_FP16_FP32", "ACC_FP32_FP32", "ACC_FP16", "GRAN_PER_BLOCK",
    "GRAN_PER_WARP", "GRAN_PER_THREAD", "default_sm_scale", "quantize_kv_head",
    "quantize_q_head", "scores", "attend_head", "sage_attention", "sage_attention_varlen",
    "attention_fp64", "round_float", "to_fp16", "to_bf16",
]


def default_sm_scale(head_dim):
    """§4.1: sm_scale=None means 1/sqrt(head_dim) of the caller's (unpadded) head_dim."""
    return float(np.float32(1.0 / np.sqrt(np.float64(head_dim))))


def sigma_p(accum):
    """Scale of P before its E4M3 rounding: 448 in every supported accumulation mode."""
    if accum == ACC_FP16:
        raise NotImplementedError("pure fp16 P·V accumulation is not supported")
    if accum not in (ACC_FP32, ACC_FP16_FP32, ACC_FP32_FP32):
        raise ValueError("unknown accumulation mode")
    return 448.0


def round_float(x, sig_bits, min_normal_exp, max_finite):
    """Round float64 values to a binary format with `sig_bits` significand bits, RNE."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex.astype(np.int64) - 1, min_normal_exp)
    qexp = e - (sig_bits - 1)
    r = np.ldexp(np.rint(np.ldexp(a, -qexp)), qexp)
    r = np.where(r > max_finite, np.inf, r)
    return np.copysign(r, x)


def to_fp16(x):
    return round_float(x, 11, -14, 65504.0)


def to_bf16(x):
    return round_float(x, 8, -126, float.fromhex("0x1.fep127"))


# --------------------------------------------------------------------------- stages 1-3
def quantize_kv_head(k, v, gran, smooth_k, smooth_v, pv="fp8"):
    """Stages 1-3 for one KV head: k, v float32 [Nk, d]. pv="fp16" keeps V' in fp16;
    pv="fp4" quantises K' and V' to two-level FP4 (oracle/fp4.py)."""
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    d = k.shape[1]
    kbar = fixed_point_mean(k) if smooth_k else np.zeros(d, np.float32)
    vbar = fixed_point_mean(v) if smooth_v else np.zeros(d, np.float32)
    ks = smooth(k, kbar)
    vs = smooth(v, vbar)
    if pv == "fp4":
        kq = fp4_group_quant(ks, K_GROUP[gran])
        vq = fp4_channel_quant(vs)
        return dict(kbar=kbar, vbar=vbar, k_smoothed=ks, v_smoothed=vs, k4=kq["carrier"],
                    sk=kq["scales"], k_codes=kq["codes"], k_block_scales=kq["block_scales"],
                    v4=vq["carrier"], sv=vq["scales"], v_codes=vq["codes"],
                    v_block_scales=vq["block_scales"], pv="fp4")
    k8, sk = int8_group_quant(ks, K_GROUP[gran])
    if pv == "fp16":
        return dict(kbar=kbar, vbar=vbar, k_smoothed=ks, v_smoothed=vs, k8=k8, sk=sk,
                    v16=to_fp16(vs), pv="fp16")
    if pv != "fp8":
        raise ValueError("pv must be 'fp8', 'fp16' or 'fp4'")
    v8, sv = fp8_channel_quant(vs)
    return dict(kbar=kbar, vbar=vbar, k_smoothed=ks, v_smoothed=vs, k8=k8, sk=sk, v8=v8, sv=sv,
                pv="fp8")


def quantize_q_head(q, gran, pv="fp8"):
    if pv == "fp4":
        qq = fp4_group_quant(np.asarray(q, np.float32), Q_GROUP[gran])
        return dict(q4=qq["carrier"], sq=qq["scales"], q_codes=qq["codes"],
                    q_block_scales=qq["block_scales"])
    q8, sq = int8_group_quant(np.asarray(q, np.float32), Q_GROUP[gran])
    return dict(q8=q8, sq=sq)


# --------------------------------------------------------------------------- steps 4-10
def scores(q8, k8):
    """Step 4 alone: S = Q8 · K8^T as exact int64 (the INT32 score contract)."""
    return np.asarray(q8, np.int64) @ np.asarray(k8, np.int64).T


def attend_head(q, kvq, *, gran, sm_scale, is_causal, accum, rows=None, qq=None,
                bypass_quant=False, row_chunk=512, p_max="final", key_tile=KEY_TILE):
    """Steps 4-10 for one query head against one quantised KV head.

    q: float32 [Nq, d] (original values, used for Q quantisation and the LSE term);
    kvq: output of quantize_kv_head; rows: query rows to compute (default all).
    bypass_quant replaces every code by the value it encodes (scales 1, P unrounded):
    the result must then equal exact attention, which pins the non-quantising steps;
    bypass_quant="qk" bypasses only the Q/K codes (P and V keep their P·V format).
    p_max: "final" (P~ against the row's maximum over all keys) or "running" (the online
    form: P~ against the maximum of the key tiles seen so far, accumulator rescaled);
    key_tile: keys per tile of the online form.
    Returns dict(o=float64 [R, d] before output rounding, lse=float64 [R]).
    """
    if p_max not in ("final", "running"):
        raise ValueError("p_max must be 'final' or 'running'")
    if key_tile < 1:
        raise ValueError("key_tile must be positive")
    q = np.asarray(q, np.float32)
    nq, d = q.shape
    nk = kvq["k_smoothed"].shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    pv16 = kvq.get("pv") == "fp16"
    pv4 = kvq.get("pv") == "fp4"
    sig = sigma_p(accum)       # raises for pure fp16 accumulation or an unknown mode
    if pv16:
        sig = 1.0              # fp16 P needs no scaling into its format's range
    if pv4:
        sig = 448.0 * 6.0      # P's carrier is ~6 · 448 p
    if bypass_quant is True:
        qv = q.astype(np.float64)
        sq_row = np.ones(nq)
        kv = kvq["k_smoothed"].astype(np.float64)
        sk_key = np.ones(nk)
        vd = kvq["v_smoothed"].astype(np.float64)
        sv = np.ones(d)
    elif bypass_quant == "qk":
        qv = q.astype(np.float64)
        sq_row = np.ones(nq)
        kv = kvq["k_smoothed"].astype(np.float64)
        sk_key = np.ones(nk)
    else:
        if qq is None:
            qq = quantize_q_head(q, gran, pv="fp4" if pv4 else "fp8")
        if pv4:
            # carriers ≈ 6 x / g: the score scale carries g_q g_k / 36
            qv = qq["q4"]
            sq_row = qq["sq"].astype(np.float64)[np.arange(nq) // Q_GROUP[gran]] / 6.0
            kv = kvq["k4"]
            sk_key = kvq["sk"].astype(np.float64)[np.arange(nk) // K_GROUP[gran]] / 6.0
        else:
            qv = qq["q8"].astype(np.float64)
            sq_row = qq["sq"].astype(np.float64)[np.arange(nq) // Q_GROUP[gran]]
            kv = kvq["k8"].astype(np.float64)
            sk_key = kvq["sk"].astype(np.float64)[np.arange(nk) // K_GROUP[gran]]
    if bypass_quant is not True:
        if pv4:
            vd = kvq["v4"]
            sv = kvq["sv"].astype(np.float64) / 6.0
        elif pv16:
            vd = kvq["v16"].astype(np.float64)
            sv = np.ones(d)
        else:
            vd = e4m3_decode(kvq["v8"])
            sv = kvq["sv"].astype(np.float64)
    vbar = kvq["vbar"].astype(np.float64)
    kbar = kvq["kbar"].astype(np.float64)

    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    keys = np.arange(nk)
    for c0 in range(0, len(rows), row_chunk):
        r = rows[c0:c0 + row_chunk]
        s = qv[r] @ kv.T                                   # step 4 (exact for integer codes)
        t = s * (sq_row[r][:, None] * sk_key[None, :] * sm_scale)  # step 5
        if is_causal:
            t = np.where(keys[None, :] <= r[:, None], t, -np.inf)

        def quantise_p(p):                                 # step 7
            if bypass_quant is True:
                return p * sig
            if pv16:
                return to_fp16(p)
            if pv4:
                return fp4_p(p, 448.0)
            return e4m3_decode(e4m3_encode(p * sig))

        if p_max == "final":
            m = t.max(axis=1)                              # step 6
            p = np.exp(t - m[:, None])
            l = p.sum(axis=1)
            acc = quantise_p(p) @ vd                       # steps 7-8
        else:
            # steps 6-8 in the online form, one 128-key tile at a time
            m = np.full(len(r), -np.inf)
            l = np.zeros(len(r))
            acc = np.zeros((len(r), d))
            for k0 in range(0, nk, key_tile):
                tt = t[:, k0:k0 + key_tile]
                m_new = np.maximum(m, tt.max(axis=1))
                m_ref = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.exp(m - m_ref)                  # 0 while no key was seen
                p = np.exp(tt - m_ref[:, None])
                acc = acc * alpha[:, None] + quantise_p(p) @ vd[k0:k0 + key_tile]
                l = l * alpha + p.sum(axis=1)
                m = m_new
        o[c0:c0 + len(r)] = acc * sv[None, :] / (sig * l[:, None]) + vbar[None, :]  # step 9
        lse[c0:c0 + len(r)] = m + np.log(l) + sm_scale * (q[r].astype(np.float64) @ kbar)  # 10
    return dict(o=o, lse=lse)


def _check_args(hq, hkv, d, accum):
    if d < 1 or d > 128:
        raise ValueError("head_dim must be in [1, 128]")
    if hkv < 1 or hq % hkv:
        raise ValueError("query heads must be a multiple of KV heads")
    sigma_p(accum)


def sage_attention(q, k, v, *, is_causal=False, sm_scale=None, gran=GRAN_PER_WARP,
                   accum=ACC_FP32, smooth_k=True, smooth_v=False, heads=None, rows=None,
                   bypass_quant=False, pv="fp8", p_max="final", key_tile=KEY_TILE):
    """Dense forward on canonical float32 arrays q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d].

    heads: optional list of (b, hq) pairs to compute (default all); rows: optional query
    rows (same for every computed head). Returns dict with o [B, Hq, R, d] and lse
    [B, Hq, R] (NaN for heads not computed) and the per-head quantised tensors.
    """
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    b_, hq, nq, d = q.shape
    hkv, nk = k.shape[1], k.shape[2]
    _check_args(hq, hkv, d, accum)
    if nk == 0:
        raise ValueError("attention over zero keys is undefined")
    if sm_scale is None:
        sm_scale = default_sm_scale(d)
    group = hq // hkv
    heads = [(b, h) for b in range(b_) for h in range(hq)] if heads is None else heads
    nr = nq if rows is None else len(rows)
    o = np.full((b_, hq, nr, d), np.nan)
    lse = np.full((b_, hq, nr), np.nan)
    kvcache, qcache = {}, {}
    for (b, h) in heads:
        key = (b, h // group)
        if key not in kvcache:
            kvcache[key] = quantize_kv_head(k[b, h // group], v[b, h // group], gran,
                                            smooth_k, smooth_v, pv=pv)
        qcache[(b, h)] = quantize_q_head(q[b, h], gran, pv="fp4" if pv == "fp4" else "fp8")
        res = attend_head(q[b, h], kvcache[key], gran=gran, sm_scale=sm_scale,
                          is_causal=is_causal, accum=accum, rows=rows, qq=qcache[(b, h)],
                          bypass_quant=bypass_quant, p_max=p_max, key_tile=key_tile)
        o[b, h] = res["o"]
        lse[b, h] = res["lse"]
    return dict(o=o, lse=lse, kv=kvcache, q=qcache, sm_scale=sm_scale)


def sage_attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, **kw):
    """Variable-length forward on packed float32 q [Tq, Hq, d], k/v [Tk, Hkv, d].

    Sequence b spans tokens [cu[b], cu[b+1]); smoothing means, quantisation groups and
    the causal mask all restart per sequence. Returns o [Tq, Hq, d] and lse [Hq, Tq].
    """
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    cq = np.asarray(cu_seqlens_q, np.int64)
    ck = np.asarray(cu_seqlens_k, np.int64)
    tq, hq, d = q.shape
    o = np.full((tq, hq, d), np.nan)
    lse = np.full((hq, tq), np.nan)
    per_seq = []
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            per_seq.append(None)
            continue
        qs = q[q0:q1].transpose(1, 0, 2)[None]
        ks = k[k0:k1].transpose(1, 0, 2)[None]
        vs = v[k0:k1].transpose(1, 0, 2)[None]
        res = sage_attention(qs, ks, vs, **kw)
        o[q0:q1] = res["o"][0].transpose(1, 0, 2)
        lse[:, q0:q1] = res["lse"][0]
        per_seq.append(res)
    return dict(o=o, lse=lse, per_seq=per_seq)


# --------------------------------------------------------------------------- fp64 reference
def attention_fp64(q, k, v, sm_scale, is_causal, rows=None):
    """Exact softmax(q k^T · sm_scale) v for one head, float64. Returns (o, lse)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, np.int64)
    t = (q[rows] @ k.T) * sm_scale
    if is_causal:
        t = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None], t, -np.inf)
    m = t.max(axis=1)
    p = np.exp(t - m[:, None])
    l = p.sum(axis=1)
    return (p @ v) / l[:, None], m + np.log(l)
