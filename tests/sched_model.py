"""A plain Python statement of the tensor-core path's automatic work schedule.

The schedule decides which cluster sweeps which 128-key steps of which 128-row tile; it is
host logic of the library's own design, not part of the attention the oracle defines, so
this model is written from the rules the kernel source documents:

  * tiles are listed longest first: sequences ranked by the key steps of their last tile
    (ties by index), tiles sequence by sequence (tree mask) or from the last tile index
    down with sequences ranked within each (causal mask);
  * R = tiles // clusters rounds of whole tiles, dealt in list order and alternating
    direction; with the tree mask and at most 1024 sequences (a list sorted longest first)
    the last three rounds deal their tiles instead to the clusters ranked by the key steps
    they hold (ties by index);
  * the tiles left over are cut into ceil(steps / L) pieces of about equal length, L the
    smallest length, at least max(4, ceil(longest / 8)), for which the pieces number at most
    the clusters; piece k goes to the k-th least-loaded cluster (sorted lists) or to
    cluster k;
  * each cluster's items lie consecutively, its whole tiles in round order and its piece
    last; the pieces of a split tile take consecutive partial-result slots, and the split
    tiles are listed in tile order for the merge.

``schedule`` returns the arrays the preparation kernel writes: the item records, the list
starts (with the numbers of items, of slots and of split tiles appended), the slot records
and the split-tile records.
"""
from __future__ import annotations

ROWS = 128
STEP = 128
MIN_PIECE = 4
MAX_PIECES = 8
MAX_RANKED = 1024
DEALT_ROUNDS = 3


def tile_steps(P, t, Q, H, causal, max_prefix, seq_cap):
    kv = P + Q
    if P < 0 or P > max_prefix or kv > seq_cap:
        return 0
    kend = kv
    if causal:
        hi = ((t + 1) * ROWS - 1) // H
        kend = P + min(hi, Q - 1) + 1
    return (kend + STEP - 1) // STEP


def schedule(prefix_len, Q, H, causal, max_prefix, seq_cap, ncl):
    B = len(prefix_len)
    T = (Q * H + ROWS - 1) // ROWS
    n_tiles = B * T

    def steps(b, t):
        return tile_steps(int(prefix_len[b]), t, Q, H, causal, max_prefix, seq_cap)

    if B <= MAX_RANKED:
        last = [steps(b, T - 1) for b in range(B)]
        order = sorted(range(B), key=lambda b: (-last[b], b))
    else:
        order = list(range(B))

    def tile_at(pos):
        if causal:
            return order[pos % B], T - 1 - pos // B
        return order[pos // T], pos % T

    R = n_tiles // ncl
    nd = R * ncl
    nr = n_tiles - nd
    dealt = not causal and B <= MAX_RANKED
    r0 = max(0, R - DEALT_ROUNDS) if dealt else R
    load = [0] * ncl
    cluster_of = [0] * nd

    def ranked():
        return sorted(range(ncl), key=lambda c: (load[c], c))

    for r in range(R):
        by_rank = ranked() if r >= r0 else [ncl - 1 - i if r & 1 else i for i in range(ncl)]
        for i in range(ncl):
            pos = r * ncl + i
            c = by_rank[i]
            load[c] += steps(*tile_at(pos))
            cluster_of[pos] = c
    by_rank = ranked() if dealt else list(range(ncl))

    rs = [steps(*tile_at(nd + i)) for i in range(nr)]
    mx = max(rs, default=0)
    lo = max(MIN_PIECE, (mx + MAX_PIECES - 1) // MAX_PIECES)
    hi = max(lo, mx)

    def count(length):
        return sum(max(1, (s + length - 1) // length) for s in rs)

    length = next((L for L in range(lo, hi) if count(L) <= ncl), hi)
    k = [max(1, (s + length - 1) // length) for s in rs]
    su, sbase, n_pieces, n_slots = [], [], 0, 0
    for ki in k:
        su.append(n_pieces)
        sbase.append(n_slots)
        n_pieces += ki
        n_slots += ki if ki > 1 else 0
    assert n_pieces <= ncl

    has_piece = [False] * ncl
    for j in range(n_pieces):
        has_piece[by_rank[j]] = True
    off, run = [], 0
    for c in range(ncl):
        off.append(run)
        run += has_piece[c]
    splits = [(*tile_at(nd + i), k[i], sbase[i]) for i in range(nr) if k[i] > 1]
    cl_start = [c * R + off[c] for c in range(ncl)] + [nd + n_pieces, n_slots, len(splits)]

    items = [None] * (nd + n_pieces)
    slot_info = [None] * n_slots
    for pos in range(nd):
        r = pos // ncl
        b, t = tile_at(pos)
        c = cluster_of[pos]
        items[c * R + off[c] + r] = (b, t, 0, steps(b, t), int(prefix_len[b]), 1, -1, -1)
    for j in range(n_pieces):
        i = max(x for x in range(nr) if su[x] <= j)
        p = j - su[i]
        b, t = tile_at(nd + i)
        ns, np_ = rs[i], k[i]
        s0, s1 = p * ns // np_, (p + 1) * ns // np_
        slot = sbase[i] + p if np_ > 1 else -1
        base = sbase[i] if np_ > 1 else -1
        c = by_rank[j]
        items[c * R + off[c] + R] = (b, t, s0, s1, int(prefix_len[b]), np_, slot, base)
        if slot >= 0:
            slot_info[slot] = (b, t, np_, base)
    return items, cl_start, slot_info, splits


def cluster_steps(items, cl_start, ncl):
    """Key steps each cluster sweeps, from the item lists."""
    return [sum(items[k][3] - items[k][2] for k in range(cl_start[c], cl_start[c + 1]))
            for c in range(ncl)]
