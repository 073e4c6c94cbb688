"""Float64 CPU oracle for tree-verify MLA-absorb attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may import this
package.  The product path (the CUDA library and its binding) never imports, links or
runs anything here, and this package imports nothing from the product.

The arithmetic lives in ``tv_oracle.c`` (plain C, float64, OpenMP over query rows); this
module only builds it with gcc and marshals numpy arrays into it.  Page citations are in
the C file's header:
  "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA Inference Engine"
  "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA Attention Kernel"
  "The Golden Reference: A Pivotal Moment in Building a Native DDTree Inference Engine"

Every function here is pinned by ``tests/test_oracle_*.py`` against closed forms, brute
force, library routines and hand-worked examples (see the design notes for the list).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tv_oracle.c")
_SRC_TREE = os.path.join(_HERE, "tree_oracle.c")
_SOURCES = {"tv": _SRC, "tree": _SRC_TREE}
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]

OK, ERR_INVALID_ARG, ERR_INVALID_TREE, ERR_UNSUPPORTED = 0, -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into liboracle.so next to them (gcc, OpenMP, no FP
    contraction)."""
    newest = max(os.path.getmtime(f) for f in _SOURCES.values())
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *_CFLAGS, *_SOURCES.values(), "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.tvo_visibility.argtypes = [P, i32, i32, P, P, P]
    lib.tvo_rope_neox.argtypes = [P, P, i32, i32, i32, i32, P, P, dbl, i32]
    lib.tvo_scatter_tree_kpe.argtypes = [P, i32, i32, i32, P, i64, P, i32, i32, i64, P]
    lib.tvo_verify_attn.argtypes = [i32, i32, i32, i32, i32, dbl, P, P, P, i64, P, i64,
                                    P, i32, i32, i64, P, P, P, i32, P, P, i32]
    lib.tvo_bf16_round.argtypes = [ctypes.c_float]
    lib.tvo_bf16_round.restype = ctypes.c_float
    lib.tvo_max_threads.restype = ctypes.c_int
    lib.tvo_set_threads.argtypes = [i32]
    lib.tro_argmax_rows.argtypes = [P, i64, i64, i64, P]
    lib.tro_tree_accept.argtypes = [P, P, P, i32, i32, P, P, P]
    lib.tro_compact_kv.argtypes = [P, i64, P, i64, i32, i32, P, i32, i32, i64, P, P, P, i32,
                                   i32, P]
    lib.tro_build_tree.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def compile_variant(src_text: str, out_path: str, which: str = "tv") -> str:
    """Compile the oracle with an edited copy of one of its sources (``which``: "tv" for
    tv_oracle.c, "tree" for tree_oracle.c); used by tests that plant a mistake in the
    oracle to show that the pins catch it.  Returns the library path."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    others = [v for k, v in _SOURCES.items() if k != which]
    subprocess.run(["gcc", *_CFLAGS, src, *others, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text(which: str = "tv") -> str:
    with open(_SOURCES[which]) as f:
        return f.read()


class use_library:
    """Context manager: route this module's functions to another compiled oracle."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} failed with status {rc}")


def max_threads() -> int:
    return int(_load().tvo_max_threads())


def set_threads(n: int) -> None:
    """Threads of the oracle's later OpenMP regions (for timing only)."""
    _load().tvo_set_threads(int(n))


def visibility(parent, want_anc=True):
    """parent [B,Q] int32 -> (vis [B,Q,Q] uint8, depth [B,Q] int32, anc [B,Q] uint64|None).

    Raises OracleError(status) on an invalid tree (status -2) or Q > 64 with anc (-3).
    """
    parent = _c(parent, np.int32)
    B, Q = parent.shape
    vis = np.zeros((B, Q, Q), np.uint8)
    depth = np.zeros((B, Q), np.int32)
    anc = np.zeros((B, Q), np.uint64) if want_anc else None
    rc = _load().tvo_visibility(_ptr(parent), B, Q, _ptr(vis), _ptr(depth), _ptr(anc))
    if rc != OK:
        err = OracleError(f"visibility failed with status {rc}")
        err.status = rc
        raise err
    return vis, depth, anc


def rope_neox(x, prefix_len, depth, base=10000.0, out_bf16=False):
    """x [B,Q,n_heads,d_rope] float32 -> rotated float32 (bf16-rounded if out_bf16)."""
    x = _c(x, np.float32)
    B, Q, NH, D = x.shape
    y = np.empty_like(x)
    rc = _load().tvo_rope_neox(_ptr(x), _ptr(y), B, Q, NH, D, _ptr(_c(prefix_len, np.int32)),
                               _ptr(_c(depth, np.int32)), float(base), int(bool(out_bf16)))
    _check(rc, "rope_neox")
    return y


def scatter_tree_kpe(kpe_tree_rot, k_pe_cache, prefix_len, page_table=None, page_size=64,
                     kv_stride_b=0):
    """Return a copy of k_pe_cache [rows, DR] with rotated tree rows written at P_b + i."""
    kpe_tree_rot = _c(kpe_tree_rot, np.float32)
    B, Q, D = kpe_tree_rot.shape
    out = np.array(k_pe_cache, dtype=np.float32, copy=True, order="C")
    pt = None if page_table is None else _c(page_table, np.int32)
    maxp = 0 if pt is None else pt.shape[1]
    rc = _load().tvo_scatter_tree_kpe(_ptr(kpe_tree_rot), B, Q, D, _ptr(out), out.shape[1],
                                      _ptr(pt), int(page_size), int(maxp), int(kv_stride_b),
                                      _ptr(_c(prefix_len, np.int32)))
    _check(rc, "scatter_tree_kpe")
    return out


def verify_attn(q_latent, q_pe, c_kv, k_pe, prefix_len, vis, scale, page_table=None,
                page_size=64, kv_stride_b=0, seqs=None, nthreads=0):
    """Masked absorbed-MLA attention in float64.

    q_latent [B,Q,H,DL], q_pe [B,Q,H,DR] (rotated), c_kv [rows,DL], k_pe [rows,DR],
    vis [B,Q,Q] uint8.  Returns (out [B,Q,H,DL] float64, lse [B,Q,H] float64); with
    ``seqs`` only those sequences are computed (others stay NaN).
    """
    q_latent = _c(q_latent, np.float32)
    q_pe = _c(q_pe, np.float32)
    c_kv = _c(c_kv, np.float32)
    k_pe = _c(k_pe, np.float32)
    B, Q, H, DL = q_latent.shape
    DR = q_pe.shape[-1]
    pt = None if page_table is None else _c(page_table, np.int32)
    maxp = 0 if pt is None else pt.shape[1]
    out = np.full((B, Q, H, DL), np.nan, np.float64)
    lse = np.full((B, Q, H), np.nan, np.float64)
    sel = None if seqs is None else _c(seqs, np.int32)
    rc = _load().tvo_verify_attn(
        B, H, Q, DL, DR, float(scale), _ptr(q_latent), _ptr(q_pe), _ptr(c_kv),
        c_kv.shape[1], _ptr(k_pe), k_pe.shape[1], _ptr(pt), int(page_size), int(maxp),
        int(kv_stride_b), _ptr(_c(prefix_len, np.int32)), _ptr(_c(vis, np.uint8)),
        _ptr(sel), 0 if sel is None else len(sel), _ptr(out), _ptr(lse), int(nthreads))
    _check(rc, "verify_attn")
    return out, lse


def bf16_round(x):
    """Elementwise round-to-nearest-even of float32 values to bf16 (slow; for pins)."""
    lib = _load()
    x = np.asarray(x, np.float32)
    return np.array([lib.tvo_bf16_round(float(v)) for v in x.ravel()], np.float32).reshape(x.shape)


def tree_verify_step(inp, seqs=None, nthreads=0):
    """The whole hot path on the CPU, from raw synthetic inputs.

    visibility -> RoPE(q_pe) -> RoPE(tree k_pe) written into a copy of the cache ->
    attention.  ``inp`` is the dict made by the synthetic-input generator.  Returns a dict
    with vis, depth, anc, q_pe_rot, k_pe_cache (after the tree rows were written), out, lse.
    """
    bf16 = inp["kv_dtype"] == "bf16"
    q_bf16 = inp["q_dtype"] == "bf16"
    vis, depth, anc = visibility(inp["parent"], want_anc=inp["Q"] <= 64)
    P = inp["prefix_len"]
    q_pe_rot = rope_neox(inp["q_pe"], P, depth, inp["rope_base"], out_bf16=q_bf16)
    kt = inp["kpe_tree"][:, :, None, :]
    kpe_rot = rope_neox(kt, P, depth, inp["rope_base"], out_bf16=bf16)[:, :, 0, :]
    k_pe_cache = scatter_tree_kpe(kpe_rot, inp["k_pe"], P, inp.get("page_table"),
                                  inp["page_size"], inp["kv_stride_b"])
    out, lse = verify_attn(inp["q_latent"], q_pe_rot, inp["c_kv"], k_pe_cache, P, vis,
                           inp["scale"], inp.get("page_table"), inp["page_size"],
                           inp["kv_stride_b"], seqs=seqs, nthreads=nthreads)
    return dict(vis=vis, depth=depth, anc=anc, q_pe_rot=q_pe_rot, kpe_tree_rot=kpe_rot,
                k_pe_cache=k_pe_cache, out=out, lse=lse)


# ---- greedy tree acceptance and post-verify compaction (tree_oracle.c) --------------

def argmax_rows(logits):
    """logits [..., V] float32 -> int32 argmax of every row (smallest index on ties)."""
    x = _c(logits, np.float32)
    V = x.shape[-1]
    rows = x.size // V
    out = np.empty(x.shape[:-1], np.int32)
    rc = _load().tro_argmax_rows(_ptr(x), rows, V, V, _ptr(out))
    _check(rc, "argmax_rows")
    return out


def tree_accept(parent, tokens, target):
    """Greedy acceptance: returns (accept_len [B], path [B,Q], new_tokens [B,Q]) int32."""
    parent = _c(parent, np.int32)
    B, Q = parent.shape
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, Q), np.int32)
    emit = np.zeros((B, Q), np.int32)
    rc = _load().tro_tree_accept(_ptr(parent), _ptr(_c(tokens, np.int32)),
                                 _ptr(_c(target, np.int32)), B, Q, _ptr(acc), _ptr(path),
                                 _ptr(emit))
    if rc != OK:
        err = OracleError(f"tree_accept failed with status {rc}")
        err.status = rc
        raise err
    return acc, path, emit


def compact_kv(c_kv, k_pe, prefix_len, path, accept_len, page_table=None, page_size=64,
               kv_stride_b=0):
    """Post-verify compaction on copies of the cache arrays: returns (c_kv, k_pe,
    new_prefix_len)."""
    ck = np.array(c_kv, dtype=np.float32, copy=True, order="C")
    kp = np.array(k_pe, dtype=np.float32, copy=True, order="C")
    path = _c(path, np.int32)
    B, Q = path.shape
    pt = None if page_table is None else _c(page_table, np.int32)
    maxp = 0 if pt is None else pt.shape[1]
    newp = np.zeros(B, np.int32)
    rc = _load().tro_compact_kv(_ptr(ck), ck.shape[1], _ptr(kp), kp.shape[1], ck.shape[1],
                                kp.shape[1], _ptr(pt), int(page_size), int(maxp),
                                int(kv_stride_b), _ptr(_c(prefix_len, np.int32)), _ptr(path),
                                _ptr(_c(accept_len, np.int32)), B, Q, _ptr(newp))
    _check(rc, "compact_kv")
    return ck, kp, newp


def build_tree(logprobs, tokens, budget, root=None):
    """Best-first draft tree from per-depth candidates: logprobs, tokens [B, L, K] (sorted
    descending over K) -> (parent, tokens, depth) int32 [B, budget+1] and score float32."""
    lp = _c(logprobs, np.float32)
    tk = _c(tokens, np.int32)
    B, L, K = lp.shape
    Q = budget + 1
    par = np.zeros((B, Q), np.int32)
    tks = np.zeros((B, Q), np.int32)
    dep = np.zeros((B, Q), np.int32)
    sc = np.zeros((B, Q), np.float32)
    rt = None if root is None else _c(root, np.int32)
    rc = _load().tro_build_tree(_ptr(lp), _ptr(tk), _ptr(rt), B, L, K, int(budget), _ptr(par),
                                _ptr(tks), _ptr(dep), _ptr(sc))
    _check(rc, "build_tree")
    return par, tks, dep, sc
