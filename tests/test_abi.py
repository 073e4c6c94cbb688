"""Host-side checks of the C ABI (CPU only: no kernel is launched).

The library must build for sm_103a, load, and export every function include/tv.h
declares; synchronous argument validation runs on the host and needs no GPU, so the
documented error codes are checked here with placeholder (never dereferenced) pointers.
"""
import ctypes

import pytest

from speculative_decoding_tree_04_gb300 import tv


def test_header_functions_exported(tvlib):
    lib = tvlib.load()
    names = tvlib.header_functions()
    assert {"tv_build_visibility", "tv_rope_neox", "tv_verify_attn",
            "tv_verify_attn_workspace_size", "tv_status_string", "tv_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libtv.so does not export {n}"
    assert lib.tv_version() >= 100


def test_status_strings(tvlib):
    lib = tvlib.load()
    for code in range(0, -8, -1):
        assert lib.tv_status_string(code)
    assert lib.tv_status_string(-99) == b"unknown status"


FAKE = 1 << 20  # 16-byte aligned placeholder address; validation never dereferences it


def fake_args(**kw):
    a = tv.AttnArgs()
    a.struct_size = ctypes.sizeof(tv.AttnArgs)
    a.B, a.H, a.Q, a.d_latent, a.d_rope = 2, 16, 17, 512, 64
    a.scale = 0.07
    a.q_dt = a.kv_dt = tv.TV_F32
    a.q_latent = a.q_pe = a.c_kv = a.k_pe = a.prefix_len = a.anc = a.out = a.lse = FAKE
    a.ckv_row_stride, a.kpe_row_stride = 512, 64
    a.cache = tv.CacheLayout(None, 64, 0, 2112)
    a.max_prefix_len = 2048
    for k, v in kw.items():
        if k == "cache":
            a.cache = v
        else:
            setattr(a, k, v)
    return a


def path_of(a):
    return tv.load().tv_verify_attn_path(ctypes.byref(a))


def test_valid_args_resolve_to_a_path(tvlib):
    assert path_of(fake_args()) == tv.PATH_SIMT


@pytest.mark.parametrize("kw,code", [
    (dict(struct_size=8), tv.TV_ERR_INVALID_ARG),
    (dict(Q=65), tv.TV_ERR_UNSUPPORTED),
    (dict(Q=0), tv.TV_ERR_INVALID_ARG),
    (dict(H=0), tv.TV_ERR_INVALID_ARG),
    (dict(d_rope=60), tv.TV_ERR_UNSUPPORTED),
    (dict(kv_dt=tv.TV_BF16), tv.TV_ERR_UNSUPPORTED),
    (dict(out=None), tv.TV_ERR_INVALID_ARG),
    (dict(c_kv=FAKE + 4), tv.TV_ERR_INVALID_ARG),
    (dict(ckv_row_stride=500), tv.TV_ERR_INVALID_ARG),
    (dict(kpe_row_stride=66), tv.TV_ERR_INVALID_ARG),
    (dict(max_prefix_len=4000), tv.TV_ERR_INVALID_ARG),     # kv_stride_b too small
    (dict(max_prefix_len=-1), tv.TV_ERR_INVALID_ARG),
    (dict(cache=tv.CacheLayout(FAKE, 64, 0, 0)), tv.TV_ERR_INVALID_ARG),
    (dict(cache=tv.CacheLayout(FAKE, 64, 4, 0)), tv.TV_ERR_INVALID_ARG),  # 2065 > 256 rows
    (dict(path=7), tv.TV_ERR_INVALID_ARG),
    (dict(num_splits=-2), tv.TV_ERR_INVALID_ARG),
    (dict(overlap_prev=2), tv.TV_ERR_INVALID_ARG),
])
def test_attn_argument_errors(tvlib, kw, code):
    assert path_of(fake_args(**kw)) == code
    assert tv.load().tv_last_error()


def test_workspace_query_is_zero_for_invalid_args(tvlib):
    lib = tv.load()
    assert lib.tv_verify_attn_workspace_size(ctypes.byref(fake_args(Q=65))) == 0


def test_visibility_argument_errors(tvlib):
    lib = tv.load()
    assert lib.tv_build_visibility(FAKE, 2, 65, FAKE, FAKE, None, None, None) == tv.TV_ERR_UNSUPPORTED
    assert lib.tv_build_visibility(FAKE, -1, 5, FAKE, FAKE, None, None, None) == tv.TV_ERR_INVALID_ARG
    assert lib.tv_build_visibility(None, 2, 5, FAKE, FAKE, None, None, None) == tv.TV_ERR_INVALID_ARG
    assert lib.tv_build_visibility(FAKE, 2, 0, FAKE, FAKE, None, None, None) == tv.TV_ERR_INVALID_ARG


def test_rope_argument_errors(tvlib):
    lib = tv.load()
    f = lib.tv_rope_neox
    ok = dict(in_dt=0, isr=64 * 4, ish=64, out_dt=0, osr=64 * 4, osh=64, B=2, Q=3, NH=4, D=64)

    def call(**kw):
        p = dict(ok, **kw)
        return f(FAKE, p["in_dt"], p["isr"], p["ish"], FAKE, p["out_dt"], p["osr"], p["osh"],
                 None, p["B"], p["Q"], p["NH"], p["D"], FAKE, FAKE, 10000.0, None)

    assert call(D=63) == tv.TV_ERR_INVALID_ARG
    assert call(D=0) == tv.TV_ERR_INVALID_ARG
    assert call(NH=0) == tv.TV_ERR_INVALID_ARG
    assert call(ish=32) == tv.TV_ERR_INVALID_ARG       # heads overlap
    assert call(isr=100) == tv.TV_ERR_INVALID_ARG      # rows overlap
    assert call(in_dt=5) == tv.TV_ERR_INVALID_ARG
    assert call(B=0) == tv.TV_OK                        # nothing to do, nothing launched


def test_tree_accept_argument_errors(tvlib):
    lib = tv.load()
    f = lib.tv_tree_accept
    ws = lib.tv_tree_accept_workspace_size(4, 9, 163840)
    assert ws > 0 and ws % 256 == 0
    assert lib.tv_tree_accept_workspace_size(4, 65, 100) == 0

    def call(B=4, Q=9, V=163840, stride=163840, dt=tv.TV_F32, logits=FAKE, wsp=FAKE, wsb=ws):
        return f(logits, dt, V, stride, FAKE, FAKE, B, Q, None, FAKE, FAKE, FAKE, None, wsp, wsb,
                 None)

    assert call(Q=65) == tv.TV_ERR_UNSUPPORTED
    assert call(Q=0) == tv.TV_ERR_INVALID_ARG
    assert call(V=0) == tv.TV_ERR_INVALID_ARG
    assert call(stride=100) == tv.TV_ERR_INVALID_ARG          # stride < vocab
    assert call(logits=FAKE + 2) == tv.TV_ERR_INVALID_ARG      # not float-aligned
    assert call(dt=7) == tv.TV_ERR_INVALID_ARG
    assert call(wsp=None) == tv.TV_ERR_WORKSPACE
    assert call(wsb=ws - 8) == tv.TV_ERR_WORKSPACE
    assert call(wsp=FAKE + 64) == tv.TV_ERR_WORKSPACE
    assert call(B=0) == tv.TV_OK


def test_compact_kv_argument_errors(tvlib):
    lib = tv.load()
    f = lib.tv_compact_kv
    good = tv.CacheLayout(FAKE, 64, 10, 0, 6400)

    def call(dt=tv.TV_BF16, DL=512, DR=64, ck=FAKE, cache=good, Q=9):
        return f(ck, FAKE, dt, DL, DR, DL, DR, ctypes.byref(cache) if cache else None, FAKE,
                 FAKE, FAKE, 2, Q, FAKE, None, None)

    assert call(Q=65) == tv.TV_ERR_UNSUPPORTED
    assert call(cache=None) == tv.TV_ERR_INVALID_ARG
    assert call(cache=tv.CacheLayout(FAKE, 64, 10, 0, 0)) == tv.TV_ERR_INVALID_ARG  # rows
    assert call(DR=4) == tv.TV_ERR_INVALID_ARG                # 8-byte rows
    assert call(ck=FAKE + 8) == tv.TV_ERR_INVALID_ARG
    assert call(dt=9) == tv.TV_ERR_INVALID_ARG
    assert call(cache=tv.CacheLayout(FAKE, 0, 10, 0, 6400)) == tv.TV_ERR_INVALID_ARG


def test_causal_mask_allows_long_q_without_anc(tvlib):
    # prefill: Q beyond 64 and no ancestor bitsets with the causal mask
    assert path_of(fake_args(Q=4096, anc=None, mask_mode=tv.MASK_CAUSAL,
                             cache=tv.CacheLayout(None, 64, 0, 8192))) == tv.PATH_SIMT
    assert path_of(fake_args(Q=4096, mask_mode=tv.MASK_TREE,
                             cache=tv.CacheLayout(None, 64, 0, 8192))) == tv.TV_ERR_UNSUPPORTED
    assert path_of(fake_args(anc=None)) == tv.TV_ERR_INVALID_ARG       # tree mode needs anc
    assert path_of(fake_args(mask_mode=2)) == tv.TV_ERR_INVALID_ARG
    # B*Q*H must stay below 2^31
    assert path_of(fake_args(B=1 << 12, Q=1 << 14, H=64, mask_mode=tv.MASK_CAUSAL, anc=None,
                             cache=tv.CacheLayout(None, 64, 0, 1 << 15))) == tv.TV_ERR_UNSUPPORTED


def test_build_tree_argument_errors(tvlib):
    f = tv.load().tv_build_tree

    def call(B=2, L=16, K=8, budget=32):
        return f(FAKE, FAKE, None, B, L, K, budget, FAKE, FAKE, None, None, None, None)

    assert call(L=17) == tv.TV_ERR_UNSUPPORTED
    assert call(K=17) == tv.TV_ERR_UNSUPPORTED
    assert call(budget=64) == tv.TV_ERR_UNSUPPORTED
    assert call(L=2, K=2, budget=7) == tv.TV_ERR_INVALID_ARG     # only 6 nodes exist
    assert call(L=0) == tv.TV_ERR_INVALID_ARG
    assert call(budget=-1) == tv.TV_ERR_INVALID_ARG
    assert call(B=0) == tv.TV_OK
    assert f(None, FAKE, None, 2, 16, 8, 32, FAKE, FAKE, None, None, None, None) == \
        tv.TV_ERR_INVALID_ARG
