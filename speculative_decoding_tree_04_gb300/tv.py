"""Thin ctypes binding of libtv (the C ABI in include/tv.h), with the same call names.

Only argument marshalling happens here: torch tensors supply device pointers, shapes,
strides and the current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if libtv.so has not been built, or a call fails,
this module raises.

    build_visibility(parent, anc, depth, dense_mask=None, status=None)
    rope_neox(x, out, prefix_len, depth, base=10000.0, cache=None)
    verify_prologue(parent, prefix_len, q_pe_in, q_pe_out, kpe_tree, ckv_tree, c_kv, k_pe, ...)
    verify_attn(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, scale, ...)
    build_tree(logprobs, cand_tokens, budget, parent, tokens, root=None, depth=None, ...)
    tree_accept(logits, parent, tokens, accept_len, path, new_tokens, target=None, ...)
    compact_kv(c_kv, k_pe, cache, prefix_len, path, accept_len, new_prefix_len, ...)
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtv.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "tv.h")

TV_OK, TV_ERR_INVALID_ARG, TV_ERR_INVALID_TREE, TV_ERR_UNSUPPORTED = 0, -1, -2, -3
TV_ERR_CUDA, TV_ERR_TIMEOUT, TV_ERR_WORKSPACE, TV_ERR_BOUNDS = -4, -5, -6, -7
TV_F32, TV_BF16 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_TCGEN05 = 0, 1, 2
PAGED_AUTO, PAGED_STEP_MAPS, PAGED_GATHER = 0, 1, 2
MASK_TREE, MASK_CAUSAL = 0, 1


class TVError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (status {code})")
        self.status = code


class CacheLayout(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("kv_stride_b", ctypes.c_int64),
                ("num_rows", ctypes.c_int64)]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Q", ctypes.c_int32),
        ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("q_dt", ctypes.c_int), ("kv_dt", ctypes.c_int),
        ("q_latent", ctypes.c_void_p), ("q_pe", ctypes.c_void_p),
        ("c_kv", ctypes.c_void_p), ("k_pe", ctypes.c_void_p),
        ("ckv_row_stride", ctypes.c_int64), ("kpe_row_stride", ctypes.c_int64),
        ("cache", CacheLayout),
        ("prefix_len", ctypes.c_void_p),
        ("max_prefix_len", ctypes.c_int32),
        ("anc", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("path", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("paged_view", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32),
        ("overlap_prev", ctypes.c_int32),
    ]


class PrologueArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("B", ctypes.c_int32), ("Q", ctypes.c_int32), ("H", ctypes.c_int32),
        ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32),
        ("parent", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
        ("q_pe_in", ctypes.c_void_p), ("q_pe_out", ctypes.c_void_p), ("q_dt", ctypes.c_int),
        ("kpe_tree", ctypes.c_void_p), ("ckv_tree", ctypes.c_void_p),
        ("c_kv", ctypes.c_void_p), ("k_pe", ctypes.c_void_p), ("kv_dt", ctypes.c_int),
        ("ckv_row_stride", ctypes.c_int64), ("kpe_row_stride", ctypes.c_int64),
        ("cache", CacheLayout),
        ("anc", ctypes.c_void_p), ("depth", ctypes.c_void_p),
        ("rope_base", ctypes.c_double),
        ("status", ctypes.c_void_p),
    ]


_lib = None


def load():
    """Open libtv.so (built by speculative_decoding_tree_04_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libtv.so is not built ({LIB_PATH}); run "
                           "`python -m speculative_decoding_tree_04_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.tv_build_visibility.argtypes = [P, i32, i32, P, P, P, P, P]
    lib.tv_rope_neox.argtypes = [P, i32, i64, i64, P, i32, i64, i64, ctypes.POINTER(CacheLayout),
                                 i32, i32, i32, i32, P, P, dbl, P]
    lib.tv_verify_attn_workspace_size.argtypes = [ctypes.POINTER(AttnArgs)]
    lib.tv_verify_attn_workspace_size.restype = ctypes.c_size_t
    lib.tv_verify_attn_path.argtypes = [ctypes.POINTER(AttnArgs)]
    lib.tv_verify_attn_launches.argtypes = [ctypes.POINTER(AttnArgs)]
    lib.tv_verify_attn.argtypes = [ctypes.POINTER(AttnArgs), P, ctypes.c_size_t, P]
    lib.tv_verify_attn_noalloc.argtypes = [ctypes.POINTER(AttnArgs), P]
    lib.tv_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.tv_status_string.argtypes = [i32]
    lib.tv_status_string.restype = ctypes.c_char_p
    lib.tv_last_error.restype = ctypes.c_char_p
    lib.tv_version.restype = ctypes.c_int
    lib.tv_testing_set_wait_fault.argtypes = [i32, ctypes.c_uint64, P]
    lib.tv_build_tree.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, P, P]
    lib.tv_verify_prologue.argtypes = [ctypes.POINTER(PrologueArgs), P]
    lib.tv_tree_accept_workspace_size.argtypes = [i32, i32, i64]
    lib.tv_tree_accept_workspace_size.restype = ctypes.c_size_t
    lib.tv_tree_accept.argtypes = [P, i32, i64, i64, P, P, i32, i32, P, P, P, P, P, P,
                                   ctypes.c_size_t, P]
    lib.tv_compact_kv.argtypes = [P, P, i32, i64, i64, i32, i32, ctypes.POINTER(CacheLayout),
                                  P, P, P, i32, i32, P, P, P]
    _lib = lib
    return lib


def header_functions(paths=None):
    """Names of the functions the headers under include/ declare (for symbol checks)."""
    if paths is None:
        inc = os.path.dirname(HEADER)
        paths = sorted(os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h"))
    names = set()
    for path in ([paths] if isinstance(paths, str) else paths):
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tv_\w+)\s*\(", text, re.M))
    return sorted(names)


def _check(rc, what):
    if rc != TV_OK:
        lib = load()
        raise TVError(rc, f"{what}: {lib.tv_last_error().decode()}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TV_F32
    if t.dtype == torch.bfloat16:
        return TV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libtv takes CUDA tensors only")


def build_visibility(parent, anc, depth, dense_mask=None, status=None, stream=None):
    """parent [B,Q] int32 -> anc [B,Q] int64 (bit patterns of uint64), depth [B,Q] int32."""
    _need_cuda(parent, anc, depth, dense_mask, status)
    assert parent.dtype == torch.int32 and anc.dtype in (torch.int64, torch.uint64)
    assert parent.is_contiguous() and anc.is_contiguous() and depth.is_contiguous()
    B, Q = parent.shape
    rc = load().tv_build_visibility(_ptr(parent), B, Q, _ptr(anc), _ptr(depth),
                                    _ptr(dense_mask), _ptr(status), _stream(stream))
    _check(rc, "tv_build_visibility")


def make_cache(page_table=None, page_size=64, kv_stride_b=0, num_rows=0) -> CacheLayout:
    """Cache geometry; num_rows = rows of the c_kv / k_pe arrays (0 = unknown)."""
    if page_table is not None:
        _need_cuda(page_table)
        assert page_table.dtype == torch.int32 and page_table.is_contiguous()
        return CacheLayout(page_table.data_ptr(), page_size, page_table.shape[1], 0, num_rows)
    return CacheLayout(None, page_size, 0, kv_stride_b, num_rows)


def rope_neox(x, out, prefix_len, depth, base=10000.0, cache: CacheLayout | None = None,
              stream=None):
    """NeoX RoPE on x [B,Q,H,D] (or [B,Q,D] for one head) into out; depth None means row
    i sits at position prefix_len + i (a chain, as in prefill).

    Without ``cache`` out has x's shape (in place allowed).  With ``cache`` out is a cache
    array [rows, D] (row stride out.stride(0)) and row (b, i) goes to the cache slot of
    logical key prefix_len[b] + i.
    """
    _need_cuda(x, out, prefix_len, depth)
    x4 = x if x.dim() == 4 else x.unsqueeze(2)
    B, Q, NH, D = x4.shape
    if x4.stride(-1) != 1 or out.stride(-1) != 1:
        raise ValueError("innermost dimension must be contiguous")
    isr, ish = x4.stride(1), x4.stride(2)
    if x4.stride(0) != Q * isr:
        raise ValueError("x rows must be uniformly strided over (B, Q)")
    if cache is None:
        o4 = out if out.dim() == 4 else out.unsqueeze(2)
        if o4.stride(0) != Q * o4.stride(1):
            raise ValueError("out rows must be uniformly strided over (B, Q)")
        osr, osh = o4.stride(1), o4.stride(2)
        cp = None
    else:
        osr, osh = out.stride(0), D
        cp = ctypes.byref(cache)
    rc = load().tv_rope_neox(_ptr(x), _dt(x), isr, ish, _ptr(out), _dt(out), osr, osh, cp,
                             B, Q, NH, D, _ptr(prefix_len), _ptr(depth), float(base),
                             _stream(stream))
    _check(rc, "tv_rope_neox")


def attn_args(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, scale, max_prefix_len,
              page_table=None, page_size=64, kv_stride_b=0, status=None, path=PATH_AUTO,
              num_splits=0, paged_view=PAGED_AUTO, mask_mode=MASK_TREE,
              overlap_prev=0) -> AttnArgs:
    _need_cuda(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, page_table, status)
    B, Q, H, DL = q_latent.shape
    DR = q_pe.shape[-1]
    for t in (q_latent, q_pe, prefix_len, anc, out, lse):
        if t is not None and not t.is_contiguous():
            raise ValueError("q_latent, q_pe, prefix_len, anc, out, lse must be contiguous")
    if c_kv.stride(-1) != 1 or k_pe.stride(-1) != 1:
        raise ValueError("cache rows must be contiguous")
    a = AttnArgs()
    a.struct_size = ctypes.sizeof(AttnArgs)
    a.B, a.H, a.Q, a.d_latent, a.d_rope = B, H, Q, DL, DR
    a.scale = float(scale)
    a.q_dt, a.kv_dt = _dt(q_latent), _dt(c_kv)
    a.q_latent, a.q_pe = q_latent.data_ptr(), q_pe.data_ptr()
    a.c_kv, a.k_pe = c_kv.data_ptr(), k_pe.data_ptr()
    a.ckv_row_stride, a.kpe_row_stride = c_kv.stride(0), k_pe.stride(0)
    a.cache = make_cache(page_table, page_size, kv_stride_b,
                         min(c_kv.shape[0], k_pe.shape[0]))
    a.prefix_len = prefix_len.data_ptr()
    a.max_prefix_len = int(max_prefix_len)
    a.anc = None if anc is None else anc.data_ptr()
    a.out, a.lse = out.data_ptr(), lse.data_ptr()
    a.status = None if status is None else status.data_ptr()
    a.path, a.num_splits, a.paged_view = int(path), int(num_splits), int(paged_view)
    a.mask_mode = int(mask_mode)
    a.overlap_prev = int(overlap_prev)
    return a


def workspace_size(a: AttnArgs) -> int:
    return int(load().tv_verify_attn_workspace_size(ctypes.byref(a)))


def attn_launches(a: AttnArgs) -> int:
    """Kernels one tv_verify_attn call with these arguments enqueues."""
    rc = load().tv_verify_attn_launches(ctypes.byref(a))
    if rc < 0:
        _check(rc, "tv_verify_attn_launches")
    return rc


def chosen_path(a: AttnArgs) -> int:
    rc = load().tv_verify_attn_path(ctypes.byref(a))
    if rc < 0:
        _check(rc, "tv_verify_attn_path")
    return rc


_ws_cache: dict = {}


def verify_attn_noalloc(a: AttnArgs, stream=None):
    """tv_verify_attn_noalloc on prepared arguments: the CUDA-core kernel with its split
    scratch in the library's fixed device array (no workspace, no allocation)."""
    rc = load().tv_verify_attn_noalloc(ctypes.byref(a), _stream(stream))
    _check(rc, "tv_verify_attn_noalloc")


def noalloc_scratch_bytes() -> int:
    return int(load().tv_noalloc_scratch_bytes())


def verify_attn(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, scale, max_prefix_len,
                page_table=None, page_size=64, kv_stride_b=0, status=None, path=PATH_AUTO,
                num_splits=0, workspace=None, stream=None, paged_view=PAGED_AUTO,
                mask_mode=MASK_TREE, overlap_prev=0):
    """Tree-verify attention; out [B,Q,H,DL] and lse [B,Q,H] (float32) are written.

    ``workspace`` (a CUDA uint8 tensor) is allocated through torch and cached per device
    when not given.  ``overlap_prev=1`` declares that the work queued before the call
    writes neither prefix_len nor the page table (tv_attn_args.overlap_prev)."""
    a = attn_args(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, scale,
                  max_prefix_len, page_table, page_size, kv_stride_b, status, path, num_splits,
                  paged_view, mask_mode, overlap_prev)
    need = workspace_size(a)
    if workspace is None and need > 0:
        key = q_latent.device
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=q_latent.device)
            _ws_cache[key] = ws
        workspace = ws
    wptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().tv_verify_attn(ctypes.byref(a), wptr, wbytes, _stream(stream))
    _check(rc, "tv_verify_attn")
    return a


def accept_workspace_size(B: int, Q: int, vocab: int) -> int:
    return int(load().tv_tree_accept_workspace_size(B, Q, vocab))


def tree_accept(logits, parent, tokens, accept_len, path, new_tokens, target=None,
                status=None, workspace=None, stream=None):
    """Greedy acceptance: logits [B,Q,V] (float32 or bf16, rows contiguous) -> accept_len
    [B], path [B,Q], new_tokens [B,Q] (and target [B,Q] if given), all int32.  The
    workspace (argmax keys) is allocated through torch and cached when not given."""
    _need_cuda(logits, parent, tokens, accept_len, path, new_tokens, target, status)
    B, Q, V = logits.shape
    if logits.stride(2) != 1 or logits.stride(0) != Q * logits.stride(1):
        raise ValueError("logits rows must be contiguous and uniformly strided over (B, Q)")
    for t in (parent, tokens, accept_len, path, new_tokens):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("parent, tokens and the outputs must be contiguous int32")
    need = accept_workspace_size(B, Q, V)
    if workspace is None and need > 0:
        key = ("accept", logits.device)
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=logits.device)
            _ws_cache[key] = ws
        workspace = ws
    wptr = None if workspace is None else ctypes.c_void_p(workspace.data_ptr())
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().tv_tree_accept(_ptr(logits), _dt(logits), V, logits.stride(1), _ptr(parent),
                               _ptr(tokens), B, Q, _ptr(target), _ptr(accept_len), _ptr(path),
                               _ptr(new_tokens), _ptr(status), wptr, wbytes, _stream(stream))
    _check(rc, "tv_tree_accept")


def compact_kv(c_kv, k_pe, cache: CacheLayout, prefix_len, path, accept_len, new_prefix_len,
               status=None, stream=None):
    """Post-verify compaction of the cache arrays c_kv [rows, DL] and k_pe [rows, DR] (in
    place) under ``cache`` (with num_rows set); new_prefix_len [B] int32 is written."""
    _need_cuda(c_kv, k_pe, prefix_len, path, accept_len, new_prefix_len, status)
    if c_kv.stride(-1) != 1 or k_pe.stride(-1) != 1:
        raise ValueError("cache rows must be contiguous")
    B, Q = path.shape
    rc = load().tv_compact_kv(_ptr(c_kv), _ptr(k_pe), _dt(c_kv), c_kv.stride(0), k_pe.stride(0),
                              c_kv.shape[1], k_pe.shape[1], ctypes.byref(cache),
                              _ptr(prefix_len), _ptr(path), _ptr(accept_len), B, Q,
                              _ptr(new_prefix_len), _ptr(status), _stream(stream))
    _check(rc, "tv_compact_kv")


def build_tree(logprobs, cand_tokens, budget, parent, tokens, root=None, depth=None, score=None,
               status=None, stream=None):
    """Best-first draft tree: logprobs [B,L,K] float32 (descending over K), cand_tokens
    [B,L,K] int32 -> parent, tokens [B, budget+1] int32 (depth, score optional)."""
    _need_cuda(logprobs, cand_tokens, root, parent, tokens, depth, score, status)
    B, L, K = logprobs.shape
    for t in (logprobs, cand_tokens, parent, tokens):
        if not t.is_contiguous():
            raise ValueError("tv_build_tree takes contiguous tensors")
    if logprobs.dtype != torch.float32 or cand_tokens.dtype != torch.int32:
        raise ValueError("logprobs must be float32 and cand_tokens int32")
    rc = load().tv_build_tree(_ptr(logprobs), _ptr(cand_tokens), _ptr(root), B, L, K,
                              int(budget), _ptr(parent), _ptr(tokens), _ptr(depth), _ptr(score),
                              _ptr(status), _stream(stream))
    _check(rc, "tv_build_tree")


def verify_prologue(parent, prefix_len, q_pe_in, q_pe_out, kpe_tree, ckv_tree, c_kv, k_pe,
                    cache: CacheLayout, anc, depth, base=10000.0, status=None, stream=None):
    """tv_verify_prologue: visibility, RoPE of q_pe (into q_pe_out, may be q_pe_in), RoPE of
    the draft keys into their cache slots and the append of the draft latent rows
    (ckv_tree may be None), in one launch."""
    _need_cuda(parent, prefix_len, q_pe_in, q_pe_out, kpe_tree, ckv_tree, c_kv, k_pe, anc,
               depth, status)
    B, Q, H, DR = q_pe_in.shape
    for t in (parent, prefix_len, q_pe_in, q_pe_out, kpe_tree, anc, depth):
        if not t.is_contiguous():
            raise ValueError("tv_verify_prologue takes contiguous tensors")
    a = PrologueArgs()
    a.struct_size = ctypes.sizeof(PrologueArgs)
    a.B, a.Q, a.H, a.d_rope = B, Q, H, DR
    a.d_latent = c_kv.shape[1]
    a.parent, a.prefix_len = parent.data_ptr(), prefix_len.data_ptr()
    a.q_pe_in, a.q_pe_out, a.q_dt = q_pe_in.data_ptr(), q_pe_out.data_ptr(), _dt(q_pe_in)
    a.kpe_tree = kpe_tree.data_ptr()
    a.ckv_tree = None if ckv_tree is None else ckv_tree.data_ptr()
    a.c_kv, a.k_pe, a.kv_dt = c_kv.data_ptr(), k_pe.data_ptr(), _dt(k_pe)
    a.ckv_row_stride, a.kpe_row_stride = c_kv.stride(0), k_pe.stride(0)
    a.cache = cache
    a.anc, a.depth = anc.data_ptr(), depth.data_ptr()
    a.rope_base = float(base)
    a.status = None if status is None else status.data_ptr()
    rc = load().tv_verify_prologue(ctypes.byref(a), _stream(stream))
    _check(rc, "tv_verify_prologue")
