"""Host-side planning of tv_verify_attn (CPU only: no kernel is launched).

The kernel family, the number of kernels a call enqueues and the workspace it asks for are
decided on the host from the argument struct.  These tests check the documented rules:

  * TV_PATH_AUTO takes the tensor cores for bf16 queries and cache with d_latent 512,
    d_rope 64 and at least 256 (row, head) rows, and the CUDA cores otherwise;
  * a tensor-core call enqueues work preparation + attention, plus a key gather when a
    paged cache's keys exceed 64 MB, plus the merge of split tiles unless every tile is
    forced into one piece;
  * the workspace has room for what the plan keeps there (split partial outputs, the
    gathered key copy), and a call refuses a workspace that is too small or misaligned
    before it launches anything.
"""
import ctypes

import pytest

from speculative_decoding_tree_04_gb300 import tv

FAKE = 1 << 20  # placeholder device address; planning never dereferences it


def args(B, H, Q, max_prefix, paged=False, dt=tv.TV_BF16, num_splits=0, path=tv.PATH_AUTO,
         paged_view=tv.PAGED_AUTO):
    a = tv.AttnArgs()
    a.struct_size = ctypes.sizeof(tv.AttnArgs)
    a.B, a.H, a.Q, a.d_latent, a.d_rope = B, H, Q, 512, 64
    a.scale = 0.07
    a.q_dt = a.kv_dt = dt
    a.q_latent = a.q_pe = a.c_kv = a.k_pe = a.prefix_len = a.anc = a.out = a.lse = FAKE
    a.ckv_row_stride, a.kpe_row_stride = 512, 64
    kv = max_prefix + Q
    if paged:
        pages = (kv + 63) // 64
        a.cache = tv.CacheLayout(FAKE, 64, pages, 0, B * pages * 64)
    else:
        a.cache = tv.CacheLayout(None, 64, 0, kv, B * kv)
    a.max_prefix_len = max_prefix
    a.num_splits = num_splits
    a.path = path
    a.paged_view = paged_view
    return a


def lib():
    return tv.load()


def path(a):
    return lib().tv_verify_attn_path(ctypes.byref(a))


def launches(a):
    return lib().tv_verify_attn_launches(ctypes.byref(a))


def workspace(a):
    return lib().tv_verify_attn_workspace_size(ctypes.byref(a))


def test_auto_path_by_shape_and_dtype(tvlib):
    assert path(args(32, 64, 33, 8192)) == tv.PATH_TCGEN05
    assert path(args(8, 64, 9, 4096, paged=True)) == tv.PATH_TCGEN05
    assert path(args(2, 16, 17, 2048, dt=tv.TV_F32)) == tv.PATH_SIMT
    assert path(args(1, 8, 5, 1)) == tv.PATH_SIMT            # 40 rows: too few for tiles
    assert path(args(1, 8, 5, 1, path=tv.PATH_TCGEN05)) == tv.PATH_TCGEN05
    a = args(2, 16, 17, 2048, dt=tv.TV_F32, path=tv.PATH_TCGEN05)
    assert path(a) == tv.TV_ERR_UNSUPPORTED                   # fp32 has no tensor-core path


def test_tensor_core_launch_structure(tvlib):
    # preparation (schedule) + attention + the merge of split tiles; the automatic schedule
    # may split tiles (decided on the device), a forced single piece per tile never does
    assert launches(args(32, 64, 33, 8192)) == 3
    assert launches(args(32, 64, 33, 8192, num_splits=1)) == 2
    assert launches(args(32, 64, 33, 8192, num_splits=3)) == 3
    # a paged cache reads its pages in place through per-step tensor maps; the gathered
    # key view, when asked for, adds the gather
    assert launches(args(32, 64, 33, 8192, paged=True)) == 3
    assert launches(args(32, 64, 33, 8192, paged=True, num_splits=1)) == 2
    assert launches(args(32, 64, 33, 8192, paged=True, num_splits=1,
                          paged_view=tv.PAGED_GATHER)) == 3
    # a paged cache of 8 x 4105 keys (about 38 MB) keeps per-step tensor maps: no gather
    assert launches(args(8, 64, 9, 4096, paged=True, num_splits=1)) == 2
    assert launches(args(8, 64, 9, 4096, paged=True)) == 3


def test_workspace_holds_what_the_plan_keeps_there(tvlib):
    rows = 32 * 33 * 64
    tiles = 32 * 17
    base = workspace(args(32, 64, 33, 8192))
    # automatic schedule: item records plus partial results for the pieces of split tiles
    # (room for two per cluster, 74 clusters assumed without a GPU)
    assert base >= 2 * 74 * 128 * (512 + 1) * 4
    assert base < 64 << 20
    ws2 = workspace(args(32, 64, 33, 8192, num_splits=2))
    ws4 = workspace(args(32, 64, 33, 8192, num_splits=4))
    assert ws2 >= 2 * tiles * 128 * (512 + 1) * 4 >= 2 * rows * (512 + 1) * 4
    assert ws4 >= 4 * tiles * 128 * (512 + 1) * 4 and ws4 > ws2
    one = workspace(args(32, 64, 33, 8192, num_splits=1))
    assert 0 < one < (1 << 20)                                # records only: no slots
    gathered = workspace(args(32, 64, 33, 8192, paged=True, paged_view=tv.PAGED_GATHER))
    assert gathered >= 32 * 8225 * (512 + 64) * 2             # contiguous key copy
    assert workspace(args(32, 64, 33, 8192, paged=True)) < gathered
    maps = workspace(args(8, 64, 9, 4096, paged=True, num_splits=1))
    assert maps >= 8 * ((4105 + 127) // 128) * 256            # two 128-byte maps per step
    assert maps < 8 * 4105 * (512 + 64) * 2                   # and no key copy
    for size in (base, ws2, gathered, maps, one):
        assert size % 256 == 0


@pytest.mark.parametrize("offset,short", [(128, False), (0, True)])
def test_call_refuses_a_bad_workspace_before_launching(tvlib, offset, short):
    a = args(32, 64, 33, 8192, num_splits=2)
    need = workspace(a)
    ws_bytes = need - 256 if short else need
    rc = lib().tv_verify_attn(ctypes.byref(a), ctypes.c_void_p(FAKE + offset), ws_bytes, None)
    assert rc == tv.TV_ERR_WORKSPACE
    assert lib().tv_last_error()


def test_paged_view_forces_either_form(tvlib):
    # small paged cache: per-step maps by default, the gathered key view when forced
    small = dict(B=8, H=64, Q=9, max_prefix=4096, paged=True, num_splits=1)
    assert launches(args(**small)) == 2
    assert launches(args(**small, paged_view=tv.PAGED_GATHER)) == 3
    assert workspace(args(**small, paged_view=tv.PAGED_GATHER)) >= 8 * 4224 * (512 + 64) * 2
    # large paged cache: per-step maps by default too, the gathered view when forced
    big = dict(B=32, H=64, Q=33, max_prefix=8192, paged=True, num_splits=1)
    assert launches(args(**big)) == 2
    assert launches(args(**big, paged_view=tv.PAGED_GATHER)) == 3
    assert workspace(args(**big, paged_view=tv.PAGED_STEP_MAPS)) < 32 * 8225 * 1152
    # a contiguous cache ignores the setting
    assert launches(args(32, 64, 33, 8192, paged_view=tv.PAGED_GATHER, num_splits=1)) == 2
    # out-of-range values are argument errors
    assert path(args(**small, paged_view=3)) == tv.TV_ERR_INVALID_ARG
