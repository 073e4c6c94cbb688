"""Tolerance rules of the parity tests (test infrastructure; no part of the method).

Floating-point outputs follow the verify-attention tolerance the pages quote -- "say,
1e-5 absolute and 1 % relative" ("The Precision Imperative: Validating Numerical Accuracy
in a Custom CUDA Attention Kernel", §"Why the Error Margin Matters") -- read as: pass iff
max_abs <= 1e-5 AND max_rel <= 1e-2, where rel_i = |g - o| / max(|o_i|, 1e-3 * max|o|)
(the floor keeps near-zero outputs from dominating).  Integer outputs: bit-exact.

bf16 caches must first pass max_abs <= 2e-2 against an oracle fed the same bf16-rounded
values.  At the large workloads that bound is about as large as the outputs themselves (a
softmax over ~6000 keys of N(0,1) rows has outputs of std ~0.0125), so a stricter rule,
derived from the arithmetic, is applied beside it:

  * attention output, per (sequence, node, head) row of d_latent values:
        rms(g - o) <= 2^-7 * rms(o).
    The only rounding of the bf16 tensor-core path that is not a float32 rounding is the
    one of the softmax weights p_j to bf16 before P.V: bf16 carries 8 significant bits,
    so round-to-nearest gives |delta_j| <= 2^-8.  The row sum l is taken from the
    unrounded weights, so
        g_d - o_d = sum_j w_j delta_j v_jd      (w = softmax weights),
    whose mean square over independent value columns is sum_j w_j^2 delta_j^2 <= 2^-16
    sum_j w_j^2, i.e. at most 2^-8 of o's rms; rows ruled by one key (sharp softmax)
    reach it (3.5e-3 measured), rows spread over many keys sit near 2^-8/sqrt(3).  The
    bound allows twice 2^-8.  float32 accumulation (K = 576 products, up to ~8000 keys)
    adds ~1e-6 relative; the CUDA-core path, whose weights stay float32, measures ~1e-6.
    Dropping the q_pe.k_pe term moves every score by ~0.04 and each row by ~4 % of its
    rms (5x the bound); a wrong 64-key page moves the rows of that sequence by ~10 % of
    their rms: both fail.
  * log-sum-exp: |g - o| <= 2^-12 * max(1, |o|).  Every step (dot products of 576
    products, the exponent sum, the final log) is float32: the score error of a 576-term
    sum is at most 576 * 2^-24 of the sum of |terms| (a few times |lse|), which the bound
    covers with margin.
"""
from __future__ import annotations

import numpy as np

FP32_ABS, FP32_REL, BF16_ABS = 1e-5, 1e-2, 2e-2
BF16_ROW_RMS = 2.0 ** -7
BF16_LSE_REL = 2.0 ** -12


def errors(gpu, ref, row_len=None):
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    if o.size == 0:
        return dict(max_abs=0.0, max_rel=0.0, raw_rel=0.0, n=0, row_rms=0.0, scaled=0.0)
    fin = np.isfinite(o)
    assert np.array_equal(fin, np.isfinite(g)), "non-finite pattern differs"
    row_rms = 0.0
    if row_len is not None:
        gr = g.reshape(-1, row_len)
        orr = o.reshape(-1, row_len)
        ok = np.all(np.isfinite(orr), axis=1)
        if ok.any():
            num = np.sqrt(np.mean((gr[ok] - orr[ok]) ** 2, axis=1))
            den = np.sqrt(np.mean(orr[ok] ** 2, axis=1))
            row_rms = float(np.max(num / np.maximum(den, 1e-30)))
    g, o = g[fin], o[fin]
    d = np.abs(g - o)
    floor = 1e-3 * np.max(np.abs(o)) if o.size else 0.0
    rel = d / np.maximum(np.abs(o), max(floor, 1e-300))
    raw = d / np.maximum(np.abs(o), 1e-300)
    scaled = d / np.maximum(np.abs(o), 1.0)
    return dict(max_abs=float(d.max(initial=0)), max_rel=float(rel.max(initial=0)),
                raw_rel=float(raw.max(initial=0)), n=int(o.size), row_rms=row_rms,
                scaled=float(scaled.max(initial=0)))


def assert_close(gpu, ref, dtype: str, what: str = "", row_len=None, lse=False):
    """fp32: the pages' rule.  bf16: max_abs <= 2e-2, and the stricter derived rule --
    per-row relative rms <= 2^-7 for attention outputs (``row_len`` = d_latent), or
    |g - o| <= 2^-12 max(1, |o|) for log-sum-exps (``lse=True``)."""
    e = errors(gpu, ref, row_len)
    if dtype == "fp32":
        ok = e["max_abs"] <= FP32_ABS and e["max_rel"] <= FP32_REL
    else:
        ok = e["max_abs"] <= BF16_ABS
        if row_len is not None:
            ok = ok and e["row_rms"] <= BF16_ROW_RMS
        if lse:
            ok = ok and e["scaled"] <= BF16_LSE_REL
    assert ok, f"{what}: {e}"
    return e


def ulp(x, dtype: str):
    """Spacing of the storage format at |x| (float32 or bf16)."""
    a = np.abs(np.asarray(x, np.float32))
    s32 = np.spacing(a).astype(np.float64)
    return s32 if dtype == "fp32" else s32 * 65536.0
