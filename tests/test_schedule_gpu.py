"""The tensor-core path's work schedule, read back from the workspace after a call.

The preparation kernel writes, into the call's workspace, the item records (which 128-key
steps of which 128-row tile each cluster sweeps), each cluster's list start, the records
of the partial-result slots and the list of split tiles the merge works through.  These tests compare them, entry by entry, with the plain
Python statement of the rules in ``tests/sched_model.py``, and check independently of it
that every tile's key steps are swept exactly once.  The attention inputs are zeros: the
schedule depends only on the sizes and the prefix lengths.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_04_gb300 import tv
from tests import sched_model

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def align256(n):
    return (n + 255) // 256 * 256


def clusters_from_size(total, n_tiles):
    """Clusters the plan used, from the workspace size of a contiguous-cache call (items,
    list starts and counts, two slots per cluster of records, one split-tile record per
    cluster, partial outputs and log-sum-exps)."""
    found = [c for c in range(1, 257)
             if align256((n_tiles + c) * 32) + align256((c + 3) * 4) + align256(2 * c * 16)
             + align256(c * 16) + align256(2 * c * 128 * 512 * 4) + align256(2 * c * 128 * 4)
             == total]
    assert len(found) == 1, found
    return found[0]


def run_schedule(prefix, Q, H, causal):
    dev = torch.device("cuda")
    B = len(prefix)
    max_prefix = int(max(prefix))
    stride = max_prefix + Q
    z = dict(dtype=torch.bfloat16, device=dev)
    q_latent = torch.zeros((B, Q, H, 512), **z)
    q_pe = torch.zeros((B, Q, H, 64), **z)
    c_kv = torch.zeros((B * stride, 512), **z)
    k_pe = torch.zeros((B * stride, 64), **z)
    prefix_len = torch.tensor(np.asarray(prefix, np.int32), device=dev)
    anc = None
    if not causal:  # every draft token sees itself only
        anc = (torch.ones((B, Q), dtype=torch.int64, device=dev)
               << torch.arange(Q, device=dev).view(1, Q))
    out = torch.empty((B, Q, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mode = tv.MASK_CAUSAL if causal else tv.MASK_TREE
    a = tv.attn_args(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, 0.05, max_prefix,
                     None, 64, stride, status, tv.PATH_TCGEN05, 0, tv.PAGED_AUTO, mode)
    need = tv.workspace_size(a)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    tv.verify_attn(q_latent, q_pe, c_kv, k_pe, prefix_len, anc, out, lse, 0.05, max_prefix,
                   None, 64, stride, status, tv.PATH_TCGEN05, 0, workspace=ws, mask_mode=mode)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(lse).all()
    T = (Q * H + 127) // 128
    n_tiles = B * T
    ncl = clusters_from_size(need, n_tiles)
    raw = ws.cpu().numpy()
    cl_off = align256((n_tiles + ncl) * 32)
    slot_off = cl_off + align256((ncl + 3) * 4)
    split_off = slot_off + align256(2 * ncl * 16)
    cl_start = raw[cl_off: cl_off + (ncl + 3) * 4].view(np.int32)
    n_items, n_slots, n_split = (int(x) for x in cl_start[ncl:])
    items = raw[: n_items * 32].view(np.int32).reshape(n_items, 8)
    slots = raw[slot_off: slot_off + n_slots * 16].view(np.int32).reshape(n_slots, 4)
    splits = raw[split_off: split_off + n_split * 16].view(np.int32).reshape(n_split, 4)
    return dict(ncl=ncl, cl_start=cl_start, items=items, slots=slots, splits=splits,
                stride=stride, max_prefix=max_prefix, T=T)


def check_against_model(prefix, Q, H, causal):
    g = run_schedule(prefix, Q, H, causal)
    ncl = g["ncl"]
    items, cl_start, slot_info, splits = sched_model.schedule(
        prefix, Q, H, causal, g["max_prefix"], g["stride"], ncl)
    assert g["cl_start"].tolist() == cl_start
    assert g["items"].tolist() == [list(it) for it in items]
    assert g["slots"].tolist() == [list(s) for s in slot_info]
    assert g["splits"].tolist() == [list(s) for s in splits]
    # every tile's steps swept exactly once, whatever the rules
    swept = {}
    for b, t, s0, s1, *_ in items:
        swept.setdefault((b, t), []).append((s0, s1))
    B = len(prefix)
    assert len(swept) == B * g["T"]
    for (b, t), runs in swept.items():
        runs.sort()
        want = sched_model.tile_steps(int(prefix[b]), t, Q, H, causal, g["max_prefix"],
                                      g["stride"])
        assert runs[0][0] == 0 and runs[-1][1] == want
        assert all(runs[i][1] == runs[i + 1][0] for i in range(len(runs) - 1))
    return sched_model.cluster_steps(items, cl_start, ncl)


def prefixes(B, lo, hi, seed):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=B).astype(np.int32)


@pytest.mark.parametrize("B,Q,H,lo,hi", [
    (32, 33, 64, 4096, 8192),     # 544 tiles: 7 rounds of unequal tiles, 12 left in pieces
    (8, 9, 64, 1024, 4096),       # 40 tiles: no whole round, every tile in pieces
    (76, 33, 64, 1, 600),         # 1292 tiles: 17 whole rounds, nothing left over
    (80, 33, 64, 2000, 3000),     # 68 tiles left over, one piece each
    (9, 33, 64, 0, 0),            # prefix 0: one key step per tile, one tile left over
    (5, 33, 64, 100000, 120000),  # 9 long tiles left over: at most 8 pieces each
    (1100, 1, 64, 0, 500),        # more sequences than are ranked: rounds alternate
    (120, 64, 128, 0, 1000),      # 7680 tiles: 101 rounds, the last 3 dealt by load
    # 1 to 5 whole rounds around the three dealt ones, ragged prefixes, tiles left over
    (5, 33, 64, 100, 3000), (9, 33, 64, 100, 3000), (14, 33, 64, 100, 3000),
    (18, 33, 64, 100, 3000), (23, 33, 64, 100, 3000),
])
def test_tree_schedule_matches_rules(B, Q, H, lo, hi):
    steps = check_against_model(prefixes(B, lo, hi, 40 + B), Q, H, False)
    if B <= sched_model.MAX_RANKED:
        # a round's tiles, longest first, go to the least-loaded clusters: none holds more
        # than the mean plus one whole tile and one piece
        longest = (hi + Q + 127) // 128
        assert max(steps) <= sum(steps) / len(steps) + 2 * longest


@pytest.mark.parametrize("prefix", [[0], [0, 5, 17, 300]])
def test_causal_schedule_matches_rules(prefix):
    # 4096-token prefill: 2048 tiles of growing length per sequence, rounds alternating
    # direction, the tiles left over in pieces
    check_against_model(prefix, 4096, 64, True)
