"""Pins of the tree-acceptance and compaction oracle (CPU only).

The oracle's argmax, greedy walk and compaction are checked against things other than
themselves:
  * numpy's argmax (first occurrence on ties) and planted ties;
  * brute force over every six-node tree: with distinct sibling tokens the accepted path is
    the longest root path whose every draft token equals its parent's target token;
  * closed forms on chain and star trees;
  * the invariant the pages state for the decode loop: greedy speculative output equals
    greedy autoregressive output token for token, simulated with a deterministic toy
    target model;
  * a hand-worked example (tests/golden/accept_worked_example.json);
  * compaction against an out-of-place gather/scatter in numpy, paged and contiguous.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_worked_example.json")


# ---- argmax -------------------------------------------------------------------------

def test_argmax_matches_numpy_and_takes_smallest_index_on_ties():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((37, 1001)).astype(np.float32)
    assert np.array_equal(oracle.argmax_rows(x), np.argmax(x, axis=1))
    # planted ties: the maximum appears at several indices
    y = np.round(rng.standard_normal((50, 300)) * 2).astype(np.float32)
    for r in range(50):
        m = y[r].max() + 1.0
        idx = rng.choice(300, size=rng.integers(2, 6), replace=False)
        y[r, idx] = m
    got = oracle.argmax_rows(y)
    assert np.array_equal(got, np.argmax(y, axis=1))
    for r in range(50):
        assert got[r] == np.flatnonzero(y[r] == y[r].max())[0]


# ---- greedy acceptance -------------------------------------------------------------

def _children(parent):
    ch = {i: [] for i in range(len(parent))}
    for c in range(1, len(parent)):
        ch[int(parent[c])].append(c)
    return ch


def _distinct_sibling_tokens(rng, parent, alphabet):
    """Draft tokens with distinct tokens among the children of every node."""
    tok = np.zeros(len(parent), np.int32)
    tok[0] = -5
    for node, kids in _children(parent).items():
        if kids:
            tok[kids] = rng.choice(alphabet, size=len(kids), replace=False)
    return tok


def _brute_force_accept(parent, tok, tgt):
    """Deepest node whose whole root path matches (unique with distinct siblings)."""
    Q = len(parent)
    best, best_depth = 0, 0
    for n in range(1, Q):
        chain, k = [], n
        while k != 0:
            chain.append(k)
            k = int(parent[k])
        chain.reverse()
        ok = all(tok[c] == tgt[int(parent[c])] for c in chain)
        if ok and len(chain) > best_depth:
            best, best_depth = n, len(chain)
    path = [0]
    k = best
    while k != 0:
        path.insert(1, k)
        k = int(parent[k])
    return best_depth, path


def test_brute_force_all_six_node_trees():
    rng = np.random.default_rng(2)
    trees = [np.array([-1, *c], np.int32)
             for c in itertools.product(*[range(i) for i in range(1, 6)])]
    assert len(trees) == 120
    for parent in trees:
        for _ in range(4):
            tok = _distinct_sibling_tokens(rng, parent, np.arange(5))
            tgt = rng.integers(0, 5, size=6).astype(np.int32)
            acc, path, emit = oracle.tree_accept(parent[None], tok[None], tgt[None])
            a, want = _brute_force_accept(parent, tok, tgt)
            assert acc[0] == a
            assert list(path[0, :a + 1]) == want and np.all(path[0, a + 1:] == -1)
            assert list(emit[0, :a]) == [int(tok[n]) for n in want[1:]]
            assert emit[0, a] == tgt[want[-1]] and np.all(emit[0, a + 1:] == -1)


def test_chain_accepts_up_to_first_mismatch():
    rng = np.random.default_rng(3)
    Q = 33
    parent = np.arange(-1, Q - 1, dtype=np.int32)[None]
    for cut in range(Q):
        tok = rng.integers(0, 1000, size=Q).astype(np.int32)
        tgt = np.roll(tok, -1).astype(np.int32)  # target at node i = draft token of node i+1
        if cut < Q - 1:
            tgt[cut] = tok[cut + 1] + 1             # first mismatch after node `cut`
        acc, path, emit = oracle.tree_accept(parent, tok[None], tgt[None])
        assert acc[0] == min(cut, Q - 1)
        assert list(path[0, :acc[0] + 1]) == list(range(acc[0] + 1))
        assert emit[0, acc[0]] == tgt[acc[0]]


def test_star_accepts_at_most_one_and_duplicate_siblings_take_smallest_index():
    Q = 9
    parent = np.array([-1] + [0] * (Q - 1), np.int32)[None]
    tok = np.array([0, 5, 6, 7, 6, 8, 9, 6, 1], np.int32)[None]
    tgt = np.array([6, 1, 2, 3, 4, 5, 6, 7, 8], np.int32)[None]
    acc, path, emit = oracle.tree_accept(parent, tok, tgt)
    # nodes 2, 4 and 7 all carry the root's target 6: the smallest index, 2, is accepted
    assert acc[0] == 1 and path[0, 1] == 2 and list(emit[0, :2]) == [6, tgt[0, 2]]
    tgt[0, 0] = 42                                    # nothing matches
    acc, path, emit = oracle.tree_accept(parent, tok, tgt)
    assert acc[0] == 0 and path[0, 0] == 0 and emit[0, 0] == 42


def test_invalid_tree_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.tree_accept(np.array([[-1, 1, 0]], np.int32), np.zeros((1, 3), np.int32),
                           np.zeros((1, 3), np.int32))


def _toy_next(history, V):
    """A deterministic stand-in for a greedy target model: the next token depends on the
    last two tokens and the position."""
    a = history[-1]
    b = history[-2] if len(history) > 1 else 0
    return (7 * a + 3 * b + 11 * len(history) + 1) % V


def test_speculative_output_equals_autoregressive_output():
    """[RoPE] §"The Broader Context: A Full Native Engine from Scratch": the greedy output
    of the speculative loop must match greedy autoregressive decoding token for token.
    Draft trees mix branches that follow the toy model with random ones; the targets are
    the toy model's predictions at every node.  Each step emits exactly the next A + 1
    autoregressive tokens, and no child of the last accepted node carries the token the
    model predicts there."""
    rng = np.random.default_rng(4)
    V = 50
    for trial in range(300):
        Q = int(rng.integers(1, 20))
        parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, Q)], np.int32)
        hist0 = list(rng.integers(0, V, size=3))
        tok = np.zeros(Q, np.int32)
        hist = {0: hist0}
        for i in range(1, Q):
            h = hist[int(parent[i])]
            siblings = [c for c in range(1, i) if parent[c] == parent[i]]
            taken = {int(tok[c]) for c in siblings}
            want = _toy_next(h, V)
            t = want if (rng.random() < 0.6 and want not in taken) else \
                int(rng.choice([v for v in range(V) if v not in taken]))
            tok[i] = t
            hist[i] = h + [t]
        tgt = np.array([_toy_next(hist[i], V) for i in range(Q)], np.int32)
        acc, path, emit = oracle.tree_accept(parent[None], tok[None], tgt[None])
        a = int(acc[0])
        ar, h = [], list(hist0)
        for _ in range(a + 1):
            nxt = _toy_next(h, V)
            ar.append(nxt)
            h.append(nxt)
        assert list(emit[0, :a + 1]) == ar, trial
        last = int(path[0, a])
        kids = [c for c in range(1, Q) if parent[c] == last]
        assert all(tok[c] != tgt[last] for c in kids)


def _golden_inputs():
    with open(GOLDEN) as f:
        g = json.load(f)
    Q, V = len(g["parent"]), g["V"]
    logits = np.full((Q, V), g["default_logit"], np.float32)
    for r, ent in g["logits_sparse"].items():
        for idx, val in ent.items():
            logits[int(r), int(idx)] = val
    return g, logits


def test_golden_worked_example():
    g, logits = _golden_inputs()
    ex = g["expected"]
    tgt = oracle.argmax_rows(logits)
    assert list(tgt) == ex["target"]
    parent = np.array([g["parent"]], np.int32)
    acc, path, emit = oracle.tree_accept(parent, np.array([g["tokens"]], np.int32), tgt[None])
    assert acc[0] == ex["accept_len"]
    assert list(path[0]) == ex["path"] and list(emit[0]) == ex["new_tokens"]
    P = g["prefix_len"]
    rows = P + len(g["parent"]) + 3
    c_kv = np.arange(rows * 4, dtype=np.float32).reshape(rows, 4)
    k_pe = -np.arange(rows * 2, dtype=np.float32).reshape(rows, 2)
    ck, kp, newp = oracle.compact_kv(c_kv, k_pe, np.array([P], np.int32), path, acc,
                                     kv_stride_b=rows)
    assert newp[0] == ex["new_prefix_len"]
    moved = {dst: src for src, dst in ex["moves"]}
    for r in range(rows):
        src = moved.get(r, r)
        assert np.array_equal(ck[r], c_kv[src]) and np.array_equal(kp[r], k_pe[src])


# ---- compaction --------------------------------------------------------------------

def _random_case(rng, B, Q, paged, page=16):
    parent = np.zeros((B, Q), np.int32)
    parent[:, 0] = -1
    for b in range(B):
        for i in range(1, Q):
            parent[b, i] = rng.integers(0, i)
    tok = np.zeros((B, Q), np.int32)
    for b in range(B):
        tok[b] = _distinct_sibling_tokens(rng, parent[b], np.arange(40))
    # targets follow a random root path for a random number of steps
    tgt = rng.integers(0, 40, size=(B, Q)).astype(np.int32)
    for b in range(B):
        cur = 0
        for _ in range(int(rng.integers(0, Q))):
            kids = [c for c in range(1, Q) if parent[b, c] == cur]
            if not kids:
                break
            c = int(rng.choice(kids))
            tgt[b, cur] = tok[b, c]
            cur = c
    P = rng.integers(0, 50, size=B).astype(np.int32)
    kv = P + Q
    if paged:
        npg = (kv + page - 1) // page
        perm = rng.permutation(int(npg.sum())).astype(np.int32)
        pt = np.full((B, int(npg.max())), -1, np.int32)
        off = 0
        for b in range(B):
            pt[b, :npg[b]] = perm[off:off + npg[b]]
            off += npg[b]
        rows, stride = int(npg.sum()) * page, 0
    else:
        pt, stride = None, int(kv.max()) + 3
        rows = B * stride
    c_kv = rng.standard_normal((rows, 8)).astype(np.float32)
    k_pe = rng.standard_normal((rows, 4)).astype(np.float32)
    return parent, tok, tgt, P, pt, stride, c_kv, k_pe, page


def _row(pt, page, stride, b, j):
    if pt is not None:
        return int(pt[b, j // page]) * page + j % page
    return b * stride + j


@pytest.mark.parametrize("paged", [False, True])
def test_compaction_equals_out_of_place_gather(paged):
    rng = np.random.default_rng(5 + paged)
    for _ in range(20):
        B, Q = int(rng.integers(1, 6)), int(rng.integers(1, 40))
        parent, tok, tgt, P, pt, stride, c_kv, k_pe, page = _random_case(rng, B, Q, paged)
        acc, path, emit = oracle.tree_accept(parent, tok, tgt)
        ck, kp, newp = oracle.compact_kv(c_kv, k_pe, P, path, acc, pt, page, stride)
        want_c, want_k = c_kv.copy(), k_pe.copy()
        for b in range(B):
            src = [_row(pt, page, stride, b, int(P[b]) + int(path[b, d]))
                   for d in range(1, acc[b] + 1)]
            dst = [_row(pt, page, stride, b, int(P[b]) + d) for d in range(1, acc[b] + 1)]
            gathered_c, gathered_k = c_kv[src].copy(), k_pe[src].copy()
            want_c[dst], want_k[dst] = gathered_c, gathered_k
            assert newp[b] == P[b] + 1 + acc[b]
        assert np.array_equal(ck, want_c) and np.array_equal(kp, want_k)
        # logical keys 0 .. new_prefix-1 now read prefix, root, accepted nodes in order
        for b in range(B):
            for d in range(acc[b] + 1):
                r_new = _row(pt, page, stride, b, int(P[b]) + d)
                r_old = _row(pt, page, stride, b, int(P[b]) + int(path[b, d]))
                assert np.array_equal(ck[r_new], c_kv[r_old])
