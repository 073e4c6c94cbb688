"""GPU parity of the best-first draft-tree builder (tv_build_tree) through the C ABI.

The tree is integer output decided by float32 comparisons that both sides make on the
same float32 sums in the same order, so parent arrays, tokens and depths must match the
oracle's heap algorithm bit for bit, and the scores exactly.  Budgets 4..63 (q_len up to
64), depth lists of 1..16, 1..16 candidates, planted ties; then the built tree drives the
rest of the step (visibility, RoPE, attention) against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.test_parity_gpu import check_step

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def run_build(d, budget):
    dev = "cuda"
    B = d["logprobs"].shape[0]
    lp = torch.from_numpy(d["logprobs"]).to(dev)
    tk = torch.from_numpy(d["cand_tokens"]).to(dev)
    root = torch.from_numpy(d["root"]).to(dev)
    par = torch.full((B, budget + 1), -7, dtype=torch.int32, device=dev)
    tks = torch.full_like(par, -7)
    dep = torch.full_like(par, -7)
    sc = torch.full((B, budget + 1), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tv.build_tree(lp, tk, budget, par, tks, root=root, depth=dep, score=sc, status=status)
    torch.cuda.synchronize()
    return (par.cpu().numpy(), tks.cpu().numpy(), dep.cpu().numpy(), sc.cpu().numpy(),
            int(status.item()))


def check(d, budget):
    par, tks, dep, sc, st = run_build(d, budget)
    opar, otks, odep, osc = oracle.build_tree(d["logprobs"], d["cand_tokens"], budget,
                                              root=d["root"])
    assert st == 0
    assert np.array_equal(par, opar)
    assert np.array_equal(tks, otks)
    assert np.array_equal(dep, odep)
    assert np.array_equal(sc, osc)
    return par


@pytest.mark.parametrize("B,L,K,budget", [(32, 16, 8, 32), (8, 16, 8, 8), (3, 16, 8, 4),
                                          (2, 16, 8, 16), (5, 10, 16, 63), (4, 16, 1, 16),
                                          (6, 1, 16, 16), (7, 6, 2, 63), (1, 3, 3, 39)])
def test_build_tree_parity(B, L, K, budget):
    d = synth.generate_draft(B, L, K, seed=B * 1000 + L * 10 + K)
    check(d, budget)


@pytest.mark.parametrize("K", [2, 4, 8])
def test_build_tree_with_ties(K):
    d = synth.generate_draft(9, 8, K, seed=77 + K, ties=True)
    check(d, 40)
    d["logprobs"][:] = 0.0                          # every score equal: breadth-first order
    par = check(d, 30)
    assert np.all(par[:, 1:] == (np.arange(1, 31) - 1) // K)


def test_unsorted_candidates_are_reported():
    d = synth.generate_draft(3, 4, 4, seed=5)
    d["logprobs"][1, 2] = d["logprobs"][1, 2][::-1].copy()
    _, _, _, _, st = run_build(d, 10)
    assert st == tv.TV_ERR_INVALID_ARG


def test_built_tree_drives_the_verify_step():
    """DDTree step from drafter proposals: tv_build_tree's parent array feeds the verify
    step (visibility, RoPE at P + depth, attention), which matches the oracle."""
    inp = synth.generate("cfg4_bf16")
    d = synth.generate_draft(inp["B"], 16, 8, seed=11)
    par, tks, dep, sc, st = run_build(d, inp["Q"] - 1)
    assert st == 0
    inp["parent"] = par
    step = VerifyStep(inp)
    step.run()
    g = step.results()
    assert np.array_equal(g["depth"], dep)
    check_step(inp, g, oracle.tree_verify_step(inp))
