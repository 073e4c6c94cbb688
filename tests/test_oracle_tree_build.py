"""Pins of the best-first draft-tree oracle (CPU only).

The oracle (tree_oracle.c) runs the heap algorithm: take the best candidate, push its K
children.  It is checked against:
  * brute force: every path of depth 1..L over K candidates, scored in float32 in depth
    order, sorted by (score descending, depth, rank path) -- the first `budget` paths;
  * closed forms: K = 1 gives a chain, L = 1 a star of the best candidates, and equal
    log-probabilities give the first nodes of the complete K-ary tree in breadth-first
    order (parent of node i is (i - 1) // K);
  * structure: parents come first, depth is the parent's plus one, each score is the
    parent's plus the node's log-probability, scores never increase along the output;
  * a hand-worked example (tests/golden/tree_build_worked_example.json).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_build_worked_example.json")


def sorted_logprobs(rng, B, L, K):
    p = rng.dirichlet(np.full(K + 1, 0.7), size=(B, L))[:, :, :K]   # mass left for the rest
    lp = np.log(np.maximum(p, 1e-30)).astype(np.float32)
    return -np.sort(-lp, axis=-1)


def rank_tokens(B, L, K):
    """token = 1000 * depth + rank, so that the ranks can be read back."""
    d = np.arange(1, L + 1)[None, :, None]
    k = np.arange(K)[None, None, :]
    return np.broadcast_to(1000 * d + k, (B, L, K)).astype(np.int32).copy()


def brute_force(lp, budget):
    L, K = lp.shape
    items = []
    for depth in range(1, L + 1):
        for path in itertools.product(range(K), repeat=depth):
            s = np.float32(0.0)
            for d, r in enumerate(path):
                s = np.float32(s + lp[d, r])
            items.append((-float(s), depth, path))
    items.sort()
    return [it[2] for it in items[:budget]]


def paths_of(parent, tokens):
    out = [()]
    for i in range(1, len(parent)):
        out.append(out[parent[i]] + (int(tokens[i]) % 1000,))
    return out


@pytest.mark.parametrize("L,K,budget", [(3, 3, 10), (4, 2, 15), (5, 3, 30), (2, 5, 20),
                                        (6, 2, 63), (3, 4, 40)])
def test_brute_force(L, K, budget):
    rng = np.random.default_rng(L * 100 + K)
    B = 5
    lp = sorted_logprobs(rng, B, L, K)
    tk = rank_tokens(B, L, K)
    par, tks, dep, sc = oracle.build_tree(lp, tk, budget)
    for b in range(B):
        got = paths_of(par[b], tks[b])[1:]
        assert got == brute_force(lp[b], budget), b


def test_ties_follow_depth_then_rank_path():
    rng = np.random.default_rng(9)
    L, K, budget = 4, 3, 30
    lp = sorted_logprobs(rng, 3, L, K)
    lp[:, :, 1] = lp[:, :, 0]                       # equal siblings everywhere
    lp[1, 2, :] = lp[1, 2, 0]
    tk = rank_tokens(3, L, K)
    par, tks, dep, sc = oracle.build_tree(lp, tk, budget)
    for b in range(3):
        assert paths_of(par[b], tks[b])[1:] == brute_force(lp[b], budget)


def test_closed_forms():
    rng = np.random.default_rng(3)
    # K = 1: a chain of budget nodes
    lp = sorted_logprobs(rng, 2, 9, 1)
    par, tks, dep, sc = oracle.build_tree(lp, rank_tokens(2, 9, 1), 9)
    assert np.array_equal(par, np.tile(np.arange(-1, 9), (2, 1)))
    assert np.array_equal(dep, np.tile(np.arange(10), (2, 1)))
    # L = 1: a star of the best budget candidates, in rank order
    lp = sorted_logprobs(rng, 2, 1, 12)
    par, tks, dep, sc = oracle.build_tree(lp, rank_tokens(2, 1, 12), 7)
    assert np.all(par[:, 1:] == 0) and np.array_equal(tks[:, 1:] % 1000, np.tile(np.arange(7), (2, 1)))
    # equal log-probabilities: the complete K-ary tree in breadth-first order
    for K in (2, 3, 4):
        lp = np.zeros((1, 6, K), np.float32)
        par, tks, dep, sc = oracle.build_tree(lp, rank_tokens(1, 6, K), 40)
        assert list(par[0, 1:]) == [(i - 1) // K for i in range(1, 41)]


def test_structure():
    rng = np.random.default_rng(4)
    B, L, K, budget = 6, 16, 8, 32
    lp = sorted_logprobs(rng, B, L, K)
    tk = rank_tokens(B, L, K)
    root = np.arange(B, dtype=np.int32) + 5
    par, tks, dep, sc = oracle.build_tree(lp, tk, budget, root=root)
    assert np.array_equal(tks[:, 0], root) and np.all(par[:, 0] == -1)
    for b in range(B):
        for i in range(1, budget + 1):
            p = par[b, i]
            assert 0 <= p < i
            assert dep[b, i] == dep[b, p] + 1
            rank = tks[b, i] % 1000
            assert sc[b, i] == np.float32(sc[b, p] + lp[b, dep[b, i] - 1, rank])
            assert sc[b, i] <= sc[b, i - 1] or i == 1


def test_golden_worked_example():
    with open(GOLDEN) as f:
        g = json.load(f)
    lp = np.array([g["logprobs"]], np.float32)
    L, K = lp.shape[1:]
    tk = np.array([[[10 * (d + 1) + k for k in range(K)] for d in range(L)]], np.int32)
    par, tks, dep, sc = oracle.build_tree(lp, tk, g["budget"], root=np.array([g["root_token"]]))
    ex = g["expected"]
    assert list(par[0]) == ex["parent"] and list(tks[0]) == ex["tokens"]
    assert list(dep[0]) == ex["depth"] and list(sc[0]) == ex["score"]


def test_rejects_impossible_budgets():
    with pytest.raises(oracle.OracleError):
        oracle.build_tree(np.zeros((1, 2, 2), np.float32), np.zeros((1, 2, 2), np.int32), 7)
    with pytest.raises(oracle.OracleError):
        oracle.build_tree(np.zeros((1, 17, 2), np.float32), np.zeros((1, 17, 2), np.int32), 3)
