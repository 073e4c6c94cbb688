"""The Python statement of the work schedule (tests/sched_model.py), checked on its own.

The GPU test compares the device's schedule with this model entry by entry, so the model
must itself be right: every tile's key steps swept exactly once, each cluster's list
consecutive, the pieces of a split tile on consecutive slots with one merge record per
split tile, at most one piece per cluster, and the dealt rounds no worse than the
alternating ones.  CPU only.
"""
import numpy as np
import pytest

from tests import sched_model


def check_invariants(prefix, Q, H, causal, ncl):
    max_prefix = int(max(prefix))
    seq_cap = max_prefix + Q
    items, cl_start, slot_info, splits = sched_model.schedule(
        prefix, Q, H, causal, max_prefix, seq_cap, ncl)
    B = len(prefix)
    T = (Q * H + 127) // 128
    n_items, n_slots, n_split = cl_start[ncl:]
    assert n_items == len(items) and n_slots == len(slot_info) and n_split == len(splits)
    assert cl_start[0] == 0 and all(cl_start[c] <= cl_start[c + 1] for c in range(ncl))
    # at most R whole tiles plus one piece per cluster
    R = B * T // ncl
    assert all(cl_start[c + 1] - cl_start[c] in (R, R + 1) for c in range(ncl))
    # every tile's steps swept exactly once
    swept = {}
    for b, t, s0, s1, P, np_, slot, base in items:
        assert P == prefix[b]
        swept.setdefault((b, t), []).append((s0, s1, np_, slot, base))
    assert len(swept) == B * T
    for (b, t), runs in swept.items():
        runs.sort()
        want = sched_model.tile_steps(int(prefix[b]), t, Q, H, causal, max_prefix, seq_cap)
        assert runs[0][0] == 0 and runs[-1][1] == want
        assert all(runs[i][1] == runs[i + 1][0] for i in range(len(runs) - 1))
        np_ = runs[0][2]
        assert all(r[2] == np_ for r in runs) and len(runs) == np_
        if np_ > 1:
            base = runs[0][4]
            assert [r[3] for r in runs] == list(range(base, base + np_))
            assert all(tuple(slot_info[s]) == (b, t, np_, base) for s in range(base, base + np_))
            assert (b, t, np_, base) in splits
        else:
            assert runs[0][3] == -1 and runs[0][4] == -1
    assert len(splits) == len(set(splits))
    return sched_model.cluster_steps(items, cl_start, ncl)


@pytest.mark.parametrize("seed", range(12))
def test_schedule_model_invariants(seed):
    rng = np.random.default_rng(seed)
    causal = seed % 4 == 3
    ncl = int(rng.choice([3, 16, 76]))
    if causal:
        Q, H, B = int(rng.choice([64, 200, 513])), int(rng.choice([8, 64])), int(rng.integers(1, 5))
        prefix = rng.integers(0, 300, size=B)
    else:
        Q, H, B = int(rng.choice([1, 9, 33])), int(rng.choice([16, 64])), int(rng.integers(1, 60))
        lo = int(rng.integers(0, 3000))
        prefix = rng.integers(lo, lo + 4000, size=B)
    check_invariants(prefix.astype(np.int32), Q, H, causal, ncl)


def test_dealt_rounds_even_the_loads():
    # ragged sequences of very different lengths: the longest-processing-time rounds keep
    # the busiest cluster within one whole tile and one piece of the mean
    rng = np.random.default_rng(5)
    for B in (24, 32, 48):
        prefix = rng.integers(4096, 8193, size=B).astype(np.int32)
        steps = check_invariants(prefix, 33, 64, False, 76)
        longest = (int(prefix.max()) + 33 + 127) // 128
        assert max(steps) <= np.mean(steps) + longest
