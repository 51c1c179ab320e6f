"""CPU oracle for SageAttention-style quantized attention — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the GPU path
computes, written from the method's description (pwwt.cn "SageAttention deployment
pitfalls guide", §1 "why attention is the bottleneck" for the three-stage idea, §4.1/§4.2
for the API knobs qk_quant_gran / pv_accum_dtype / smooth_k / smooth_v, §4 for
sageattn_varlen), with a stated reading wherever the guide is silent; each module's docstring
names the readings it takes.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import it. The product path
(``quantized_attention_mean_gb300``) never does: it shares no code, table or helper with
this package, and fails loudly when its CUDA library is missing.

All floating-point work that is not explicitly a quantisation step runs in float64.
The quantisation steps run in float32 exactly as the method's scale/reciprocal/round
sequence defines them, so that integer and FP8 codes can be compared bit for bit.

Parity status per function (see the pins in ``tests/test_oracle_*.py``):
  fp8.e4m3_encode / e4m3_decode          pinned (brute-force nearest-value search, spec table)
  quant.fixed_point_mean                 pinned (exact rational arithmetic)
  quant.int8_group_quant                 pinned (hand-derived cases, round-trip bound, extremes)
  quant.fp8_channel_quant                pinned (bound + extremes + brute force)
  attention.sage_attention               pinned (closed forms: Nk=1, uniform keys, constant V,
                                          causal row 0; quantisation bypass == fp64 attention;
                                          smooth_k invariance; cosine vs fp64)
  attention online form (p_max="running") pinned (one key tile: identical to the final form,
                                          FP8 and FP16 P·V; varlen == per-sequence dense;
                                          codes bypassed: exact attention, causal or not; every
                                          row's maximum in its first tile: final form to 1e-12)
  accumulation modes                     pinned (fp16+fp32, fp32+fp32 and fp32 are one
                                          arithmetic, σ_P = 448: a two-key case worked by hand
                                          from the E4M3 table, identical-key and single-key
                                          closed forms in every mode)
  fp4.e2m1_encode / e2m1_decode          pinned (value table from the field layout, brute-force
                                          nearest value with ties to the even mantissa)
  fp4.microscale_blocks / fp4_*_quant    pinned (block-step properties, a hand-worked block,
                                          reconstruction bound, lossless inputs round-trip)
  attention FP4 variant (pv="fp4")       pinned (single-key and two-key closed forms on inputs
                                          FP4 represents exactly; bypass == fp64 attention;
                                          one tile: online == final form)
  merge.merge_partials                   pinned (chunked fp64 attention merges to the unchunked
                                          result; empty parts; single part; order invariance)
"""

from . import fp4, fp8, quant, attention, merge  # noqa: F401
