"""Pins for the oracle's draft-tree visibility (CPU only).

The visibility rule -- a tree node sees its ancestor-or-self nodes -- is the mask that
"The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA Attention
Kernel" (§Context) describes for the verify kernel.  The oracle finds it by walking the
parent chain; these tests pin it to independent constructions: a boolean
transitive closure by repeated matrix products, networkx's ancestor search, and the
closed forms of chain and star trees.
"""
import itertools

import networkx as nx
import numpy as np
import pytest

import oracle


def closure_vis(parent):
    """Ancestor-or-self matrix by boolean matrix powers of the child->parent relation."""
    Q = len(parent)
    A = np.zeros((Q, Q), bool)
    for i in range(1, Q):
        A[i, parent[i]] = True
    R = np.eye(Q, dtype=bool)
    for _ in range(Q):
        R = R | ((R.astype(np.int64) @ A.astype(np.int64)) > 0)
    return R


def all_parent_arrays(Q):
    ranges = [range(i) for i in range(1, Q)]
    for combo in itertools.product(*ranges):
        yield np.array([-1, *combo], np.int32)


def test_brute_force_all_trees_q6():
    """All 1*1*2*3*4*5 = 120 topologically ordered trees with 6 nodes."""
    trees = np.stack(list(all_parent_arrays(6)))
    assert trees.shape == (120, 6)
    vis, depth, anc = oracle.visibility(trees)
    for b, par in enumerate(trees):
        R = closure_vis(par)
        assert np.array_equal(vis[b].astype(bool), R)
        assert np.array_equal(depth[b], R.sum(1) - 1)
        bits = [sum(1 << k for k in range(6) if R[i, k]) for i in range(6)]
        assert [int(x) for x in anc[b]] == bits


def test_networkx_ancestors_random_trees():
    rng = np.random.default_rng(5)
    for Q in (1, 2, 17, 33, 64):
        par = np.array([-1] + [rng.integers(0, i) for i in range(1, Q)], np.int32)
        g = nx.DiGraph()
        g.add_nodes_from(range(Q))
        g.add_edges_from((int(par[i]), i) for i in range(1, Q))
        vis, depth, anc = oracle.visibility(par[None])
        for i in range(Q):
            expect = nx.ancestors(g, i) | {i}
            got = {k for k in range(Q) if vis[0, i, k]}
            assert got == expect
            assert depth[0, i] == nx.shortest_path_length(g, 0, i)
            assert int(anc[0, i]) == sum(1 << k for k in expect)


def test_chain_is_lower_triangular():
    Q = 33
    par = np.arange(-1, Q - 1, dtype=np.int32)[None]
    vis, depth, _ = oracle.visibility(par)
    assert np.array_equal(vis[0], np.tril(np.ones((Q, Q), np.uint8)))
    assert np.array_equal(depth[0], np.arange(Q))


def test_star_sees_root_and_self():
    Q = 9
    par = np.zeros((1, Q), np.int32)
    par[0, 0] = -1
    vis, depth, _ = oracle.visibility(par)
    expect = np.eye(Q, dtype=np.uint8)
    expect[:, 0] = 1
    assert np.array_equal(vis[0], expect)
    assert np.array_equal(depth[0], np.r_[0, np.ones(Q - 1, int)])


def test_q64_top_bit():
    par = np.arange(-1, 63, dtype=np.int32)[None]
    _, _, anc = oracle.visibility(par)
    assert int(anc[0, 63]) == (1 << 64) - 1
    assert int(anc[0, 0]) == 1


@pytest.mark.parametrize("bad", [
    [0, 0, 1],        # root parent must be -1
    [-1, 1, 0],       # parent[i] must be < i
    [-1, 0, -1],      # non-root parent must be >= 0
    [-1, 0, 5],       # out of range
])
def test_invalid_trees_rejected(bad):
    with pytest.raises(oracle.OracleError) as e:
        oracle.visibility(np.array([bad], np.int32))
    assert e.value.status == oracle.ERR_INVALID_TREE


def test_q65_bitset_unsupported_but_mask_ok():
    par = np.arange(-1, 64, dtype=np.int32)[None]
    with pytest.raises(oracle.OracleError) as e:
        oracle.visibility(par, want_anc=True)
    assert e.value.status == oracle.ERR_UNSUPPORTED
    vis, depth, _ = oracle.visibility(par, want_anc=False)
    assert vis.shape == (1, 65, 65) and depth[0, 64] == 64
