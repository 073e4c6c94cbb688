"""Pins for the oracle's tree-verify attention (CPU only).

The method -- per (sequence, tree node, head), softmax attention in the absorbed latent
space over every prefix key plus the node's ancestor-or-self tree keys, returning the
softmax-weighted latent sum -- is the one described on "The Precision Imperative:
Validating Numerical Accuracy in a Custom CUDA Attention Kernel" (§Context, §"Input
Knowledge Required") and "The Golden Reference: A Pivotal Moment in Building a Native
DDTree Inference Engine" (§"The Absorb Form of MLA", §"Principled Abstraction").

Pins, none of which retypes the oracle's loop:
  * torch's scaled_dot_product_attention (float64) with a boolean mask built by networkx;
  * a chain tree equals causal attention, a root row / q_len 1 equals one decode query
    (the two degenerate cases the last page names), a star tree sees prefix+root+self;
  * zero queries give the plain mean of the visible rows and lse = ln |V|;
  * one dominant score selects its row; all-ones values give exactly 1 (weights sum to 1);
  * outputs stay inside the per-column range of the visible rows; heads are independent;
  * paged and contiguous layouts of the same data agree bit for bit;
  * a hand-worked example with closed-form weights.
"""
import json
import math
import os

import networkx as nx
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make_case(B=2, H=3, Q=6, P=(5, 0), DL=8, DR=4, seed=0, tree="random", paged=False,
              page=4):
    rng = np.random.default_rng(seed)
    parent = np.zeros((B, Q), np.int32)
    parent[:, 0] = -1
    for b in range(B):
        for i in range(1, Q):
            parent[b, i] = {"random": rng.integers(0, i), "chain": i - 1, "star": 0}[tree]
    P = np.array(P, np.int32)
    kv = P + Q
    ql = rng.standard_normal((B, Q, H, DL)).astype(np.float32)
    qr = rng.standard_normal((B, Q, H, DR)).astype(np.float32)
    logical_c = [rng.standard_normal((int(kv[b]), DL)).astype(np.float32) for b in range(B)]
    logical_k = [rng.standard_normal((int(kv[b]), DR)).astype(np.float32) for b in range(B)]
    case = dict(parent=parent, P=P, ql=ql, qr=qr, lc=logical_c, lk=logical_k, scale=0.37)
    case.update(layout(case, paged, page, rng))
    return case


def layout(case, paged, page, rng):
    """Place each sequence's logical rows into a contiguous or a shuffled paged cache."""
    lc, lk = case["lc"], case["lk"]
    B = len(lc)
    DL, DR = lc[0].shape[1], lk[0].shape[1]
    if not paged:
        S = max(len(x) for x in lc) + 3
        c = rng.standard_normal((B * S, DL)).astype(np.float32)
        k = rng.standard_normal((B * S, DR)).astype(np.float32)
        for b in range(B):
            c[b * S: b * S + len(lc[b])] = lc[b]
            k[b * S: b * S + len(lk[b])] = lk[b]
        return dict(c_kv=c, k_pe=k, page_table=None, page_size=page, kv_stride_b=S)
    npg = [(len(x) + page - 1) // page for x in lc]
    perm = rng.permutation(sum(npg)).astype(np.int32)
    pt = np.full((B, max(npg)), -1, np.int32)
    c = rng.standard_normal((sum(npg) * page, DL)).astype(np.float32)
    k = rng.standard_normal((sum(npg) * page, DR)).astype(np.float32)
    off = 0
    for b in range(B):
        pt[b, :npg[b]] = perm[off: off + npg[b]]
        off += npg[b]
        for j in range(len(lc[b])):
            row = pt[b, j // page] * page + j % page
            c[row], k[row] = lc[b][j], lk[b][j]
    return dict(c_kv=c, k_pe=k, page_table=pt, page_size=page, kv_stride_b=0)


def run_oracle(case):
    vis, _, _ = oracle.visibility(case["parent"])
    return oracle.verify_attn(case["ql"], case["qr"], case["c_kv"], case["k_pe"], case["P"],
                              vis, case["scale"], case["page_table"], case["page_size"],
                              case["kv_stride_b"])


def nx_mask(parent_row, P):
    """[Q, P+Q] boolean visibility from networkx ancestors."""
    Q = len(parent_row)
    g = nx.DiGraph()
    g.add_nodes_from(range(Q))
    g.add_edges_from((int(parent_row[i]), i) for i in range(1, Q))
    m = np.zeros((Q, P + Q), bool)
    m[:, :P] = True
    for i in range(Q):
        for k in nx.ancestors(g, i) | {i}:
            m[i, P + k] = True
    return m


def sdpa_ref(case, b, mask):
    """torch SDPA in float64 on the concatenated absorbed query/key; value = latent rows."""
    q = torch.from_numpy(np.concatenate([case["ql"][b], case["qr"][b]], -1)).double()
    k = torch.from_numpy(np.concatenate([case["lc"][b], case["lk"][b]], -1)).double()
    v = torch.from_numpy(case["lc"][b]).double()
    q = q.permute(1, 0, 2)                          # [H, Q, E]
    m = torch.from_numpy(mask)
    out = F.scaled_dot_product_attention(q, k[None].expand(q.shape[0], -1, -1),
                                         v[None].expand(q.shape[0], -1, -1),
                                         attn_mask=m, scale=case["scale"])
    scores = torch.einsum("hqe,ke->hqk", q, k) * case["scale"]
    lse = torch.logsumexp(scores.masked_fill(~m, float("-inf")), dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("tree", ["random", "chain", "star"])
def test_matches_sdpa_with_networkx_mask(paged, tree):
    case = make_case(seed=7, paged=paged, tree=tree)
    out, lse = run_oracle(case)
    for b in range(2):
        ref_o, ref_l = sdpa_ref(case, b, nx_mask(case["parent"][b], int(case["P"][b])))
        assert np.allclose(out[b], ref_o, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[b], ref_l, rtol=1e-12, atol=1e-12)


def test_chain_tree_is_causal_attention():
    case = make_case(B=1, H=2, Q=7, P=(9,), seed=3, tree="chain")
    out, lse = run_oracle(case)
    P, Q = 9, 7
    causal = np.tril(np.ones((Q, P + Q), bool), k=P)       # query i sees keys 0..P+i
    ref_o, ref_l = sdpa_ref(case, 0, causal)
    assert np.allclose(out[0], ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse[0], ref_l, rtol=1e-12, atol=1e-12)


def test_root_row_and_q1_are_single_query_decode():
    for Q in (1, 5):
        case = make_case(B=1, H=4, Q=Q, P=(11,), seed=Q)
        out, lse = run_oracle(case)
        P = 11
        q = torch.from_numpy(np.concatenate([case["ql"][0, 0], case["qr"][0, 0]], -1)).double()
        k = torch.from_numpy(np.concatenate([case["lc"][0], case["lk"][0]], -1)[:P + 1]).double()
        v = torch.from_numpy(case["lc"][0][:P + 1]).double()
        ref = F.scaled_dot_product_attention(q[:, None], k[None].expand(4, -1, -1),
                                             v[None].expand(4, -1, -1), scale=case["scale"])
        assert np.allclose(out[0, 0], ref[:, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_zero_query_is_mean_and_lse_is_log_count():
    case = make_case(seed=9)
    case["ql"][:] = 0
    case["qr"][:] = 0
    out, lse = run_oracle(case)
    for b in range(2):
        m = nx_mask(case["parent"][b], int(case["P"][b]))
        for i in range(m.shape[0]):
            rows = case["lc"][b][m[i]].astype(np.float64)
            assert np.allclose(out[b, i], rows.mean(0)[None], rtol=1e-13, atol=1e-14)
            assert np.allclose(lse[b, i], math.log(m[i].sum()), rtol=0, atol=1e-13)


def test_dominant_score_selects_row_and_ones_give_one():
    case = make_case(B=1, H=1, Q=4, P=(6,), DL=8, DR=4, seed=4, tree="chain")
    # make key 2 (a prefix key) dominate: q aligned with it, scores of others small
    case["ql"][:] = 0
    case["qr"][:] = 0
    case["lc"][0][:] *= 1e-3
    case["lk"][0][:] = 0
    case["lc"][0][2] = 0
    case["lc"][0][2, 0] = 1.0
    case["ql"][0, :, 0, 0] = 40.0 / case["scale"]
    case.update(layout(case, False, 4, np.random.default_rng(0)))
    out, lse = run_oracle(case)
    assert np.allclose(out[0, :, 0], case["lc"][0][2][None].astype(np.float64), atol=1e-15)
    assert np.allclose(lse[0, :, 0], 40.0, atol=1e-12)
    # all-ones values: weights sum to one exactly up to rounding
    for b in range(len(case["lc"])):
        case["lc"][b][:] = 1.0
    case["ql"] = np.random.default_rng(1).standard_normal(case["ql"].shape).astype(np.float32)
    case.update(layout(case, True, 4, np.random.default_rng(2)))
    out, _ = run_oracle(case)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-14)


def test_outputs_within_visible_column_range_and_heads_independent():
    case = make_case(B=2, H=4, Q=6, P=(3, 0), seed=12)
    out, lse = run_oracle(case)
    for b in range(2):
        m = nx_mask(case["parent"][b], int(case["P"][b]))
        for i in range(6):
            rows = case["lc"][b][m[i]]
            assert np.all(out[b, i] <= rows.max(0)[None] + 1e-12)
            assert np.all(out[b, i] >= rows.min(0)[None] - 1e-12)
    perm = np.array([2, 0, 3, 1])
    case2 = dict(case)
    case2["ql"] = case["ql"][:, :, perm].copy()
    case2["qr"] = case["qr"][:, :, perm].copy()
    out2, lse2 = run_oracle(case2)
    assert np.array_equal(out2, out[:, :, perm])
    assert np.array_equal(lse2, lse[:, :, perm])


def test_paged_equals_contiguous_bitwise():
    case = make_case(B=3, H=2, Q=5, P=(0, 7, 13), seed=21, paged=False)
    o1, l1 = run_oracle(case)
    case.update(layout(case, True, 4, np.random.default_rng(5)))
    o2, l2 = run_oracle(case)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "attn_worked_example.json")) as f:
        g = json.load(f)
    par = np.array([g["parent"]], np.int32)
    vis, _, _ = oracle.visibility(par)
    ql = np.array(g["q_latent"], np.float32)[None, :, None, :]
    qr = np.array(g["q_pe"], np.float32)[None, :, None, :]
    out, lse = oracle.verify_attn(ql, qr, np.array(g["c_kv"], np.float32),
                                  np.array(g["k_pe"], np.float32),
                                  np.array([g["prefix_len"]], np.int32), vis, g["scale"],
                                  kv_stride_b=len(g["c_kv"]))
    assert np.allclose(out[0, :, 0], np.array(g["expected_out"]), rtol=1e-6, atol=0)
    assert np.allclose(lse[0, :, 0], np.array(g["expected_lse"]), rtol=1e-6, atol=0)


def test_full_step_chain_equals_rope_then_causal_attention():
    """The whole step: positions P+depth, tree k_pe rows into slots P+i, then attention.

    With a chain tree depth(i) = i, so every tree key sits at RoPE position P+i and the
    step must equal causal attention with complex-multiplication RoPE applied to q_pe
    (at P+i) and to the tree k_pe rows (at P+i)."""
    from speculative_decoding_tree_04_gb300 import synth
    inp = synth.generate(B=1, H=2, Q=6, DL=16, DR=8, prefix=(10, 10), tree="chain",
                         seed=5, paged=True, page=4)
    res = oracle.tree_verify_step(inp)
    P, Q = 10, 6

    def crope(x, pos):
        h = x.shape[-1] // 2
        k = np.arange(h)
        ang = np.asarray(pos, np.float64)[..., None] * (10000.0 ** (-(2.0 * k) / x.shape[-1]))
        z = (x[..., :h].astype(np.float64) + 1j * x[..., h:]) * np.exp(1j * ang)
        return np.concatenate([z.real, z.imag], -1).astype(np.float32)

    pos = P + np.arange(Q)
    qr = crope(inp["q_pe"][0], pos[:, None])            # [Q, H, DR]
    kt = crope(inp["kpe_tree"][0], pos)                 # [Q, DR]
    pt, ps = inp["page_table"], inp["page_size"]
    rows = [pt[0, j // ps] * ps + j % ps for j in range(P + Q)]
    lc = inp["c_kv"][rows]
    lk = inp["k_pe"][rows].copy()
    lk[P:] = kt
    case = dict(ql=inp["q_latent"], qr=qr[None], lc=[lc], lk=[lk], scale=inp["scale"])
    ref_o, ref_l = sdpa_ref(case, 0, np.tril(np.ones((Q, P + Q), bool), k=P))
    assert np.allclose(res["out"][0], ref_o, rtol=1e-9, atol=1e-9)
    assert np.allclose(res["lse"][0], ref_l, rtol=1e-9, atol=1e-9)
