"""Tolerance rules of the parity tests (test infrastructure; no part of the method).

Floating-point outputs follow the verify-attention tolerance the pages quote -- "say,
1e-5 absolute and 1 % relative" ("The Precision Imperative: Validating Numerical Accuracy
in a Custom CUDA Attention Kernel", §"Why the Error Margin Matters") -- read as: pass iff
max_abs <= 1e-5 AND max_rel <= 1e-2, where rel_i = |g - o| / max(|o_i|, 1e-3 * max|o|)
(the floor keeps near-zero outputs from dominating).  bf16 caches: max_abs <= 2e-2
against an oracle fed the same bf16-rounded values.  Integer outputs: bit-exact.
"""
from __future__ import annotations

import numpy as np

FP32_ABS, FP32_REL, BF16_ABS = 1e-5, 1e-2, 2e-2


def errors(gpu, ref):
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    if o.size == 0:
        return dict(max_abs=0.0, max_rel=0.0, raw_rel=0.0, n=0)
    fin = np.isfinite(o)
    assert np.array_equal(fin, np.isfinite(g)), "non-finite pattern differs"
    g, o = g[fin], o[fin]
    d = np.abs(g - o)
    floor = 1e-3 * np.max(np.abs(o)) if o.size else 0.0
    rel = d / np.maximum(np.abs(o), max(floor, 1e-300))
    raw = d / np.maximum(np.abs(o), 1e-300)
    return dict(max_abs=float(d.max(initial=0)), max_rel=float(rel.max(initial=0)),
                raw_rel=float(raw.max(initial=0)), n=int(o.size))


def assert_close(gpu, ref, dtype: str, what: str = ""):
    e = errors(gpu, ref)
    if dtype == "fp32":
        ok = e["max_abs"] <= FP32_ABS and e["max_rel"] <= FP32_REL
    else:
        ok = e["max_abs"] <= BF16_ABS
    assert ok, f"{what}: {e}"
    return e


def ulp(x, dtype: str):
    """Spacing of the storage format at |x| (float32 or bf16)."""
    a = np.abs(np.asarray(x, np.float32))
    s32 = np.spacing(a).astype(np.float64)
    return s32 if dtype == "fp32" else s32 * 65536.0
