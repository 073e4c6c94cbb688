"""The seeded input generator against its recipe (CPU only).

Both the oracle and the CUDA path take their inputs from ``synth.generate``; these tests
pin what it draws to the workload recipe: shapes, tree rules, prefix ranges, a paged
cache whose pages are a shuffled permutation covering every live key, bf16 rounding,
the value distributions, and determinism under the seed.
"""
import math

import numpy as np
import pytest

from speculative_decoding_tree_04_gb300 import synth

SMALL = ["cfg1_fp32", "cfg2_fp32", "cfg3_fp32", "cfg3_bf16", "cfg4_bf16"]


@pytest.mark.parametrize("name", SMALL)
def test_shapes_and_sizes(name):
    w = synth.WORKLOADS[name]
    inp = synth.generate(name)
    B, H, Q, DL, DR = w["B"], w["H"], w["Q"], w["DL"], w["DR"]
    assert (inp["B"], inp["H"], inp["Q"], inp["DL"], inp["DR"]) == (B, H, Q, DL, DR)
    assert inp["parent"].shape == (B, Q) and inp["parent"].dtype == np.int32
    assert inp["prefix_len"].shape == (B,) and inp["prefix_len"].dtype == np.int32
    assert inp["q_latent"].shape == (B, Q, H, DL)
    assert inp["q_pe"].shape == (B, Q, H, DR)
    assert inp["kpe_tree"].shape == (B, Q, DR)
    assert inp["c_kv"].shape[1] == DL and inp["k_pe"].shape[1] == DR
    assert inp["c_kv"].shape[0] == inp["k_pe"].shape[0]
    assert inp["scale"] == pytest.approx(1.0 / math.sqrt(w["scale_den"]), rel=1e-7)
    assert inp["rope_base"] == 10000.0


@pytest.mark.parametrize("name", SMALL + ["cfg5_bf16"])
def test_trees_follow_the_recipe(name):
    w = synth.WORKLOADS[name]
    par = synth.generate(name, **({"DL": 8, "DR": 8, "H": 1} if name == "cfg5_bf16" else {}))["parent"]
    B, Q = par.shape
    assert np.all(par[:, 0] == -1)
    i = np.arange(1, Q)
    for b in range(B):
        p = par[b, 1:]
        assert np.all((p >= 0) & (p < i))                   # topological, one root
        kind = w["tree"]
        if kind == "mix":
            kind = "chain" if b % 2 == 1 else "random"
        if kind == "chain":
            assert np.array_equal(p, i - 1)
        elif kind == "wide":
            assert np.all(p <= np.minimum(i - 1, 3))


def test_random_parents_cover_their_range():
    # parent[i] ~ U{0..i-1}: over many sequences every allowed parent appears
    par = synth.generate(None, B=400, H=1, Q=9, DL=8, DR=8, prefix=(1, 1))["parent"]
    for i in range(1, 9):
        assert set(np.unique(par[:, i])) == set(range(i))


@pytest.mark.parametrize("name", SMALL)
def test_prefix_lengths_in_range(name):
    lo, hi = synth.WORKLOADS[name]["prefix"]
    P = synth.generate(name)["prefix_len"]
    assert np.all((P >= lo) & (P <= hi))


def test_ragged_prefixes_spread_over_the_range():
    P = synth.generate(None, B=2000, H=1, Q=2, DL=8, DR=8, prefix=(4096, 8192))["prefix_len"]
    assert P.min() < 4096 + 200 and P.max() > 8192 - 200
    assert abs(P.mean() - 6144) < 100


@pytest.mark.parametrize("name", ["cfg4_bf16"])
def test_paged_cache_is_a_shuffled_permutation_covering_live_keys(name):
    inp = synth.generate(name)
    pt, P, Q, page = inp["page_table"], inp["prefix_len"], inp["Q"], inp["page_size"]
    npg = (P.astype(np.int64) + Q + page - 1) // page
    live = np.concatenate([pt[b, :npg[b]] for b in range(inp["B"])])
    assert np.all(live >= 0)
    assert np.array_equal(np.sort(live), np.arange(live.size))          # each page once
    assert inp["c_kv"].shape[0] == live.size * page                    # no spare rows
    for b in range(inp["B"]):
        assert np.all(pt[b, npg[b]:] == -1)
    assert not np.array_equal(live, np.arange(live.size))              # shuffled


def test_contiguous_cache_geometry():
    inp = synth.generate("cfg2_fp32")
    assert inp["page_table"] is None
    kv = inp["prefix_len"].astype(np.int64) + inp["Q"]
    assert inp["kv_stride_b"] >= kv.max() and inp["kv_stride_b"] % 64 == 0
    assert inp["c_kv"].shape[0] == inp["B"] * inp["kv_stride_b"]


def test_value_distributions():
    inp = synth.generate("cfg2_fp32")
    q = inp["q_latent"].astype(np.float64)
    assert abs(q.mean()) < 0.01 and q.std() == pytest.approx(1 / math.sqrt(192), rel=0.02)
    c = inp["c_kv"].astype(np.float64)
    assert abs(c.mean()) < 0.01 and c.std() == pytest.approx(1.0, rel=0.02)
    assert np.all(np.isfinite(c)) and np.all(np.isfinite(inp["k_pe"]))


def test_bf16_values_are_representable_and_match_their_bits():
    inp = synth.generate("cfg3_bf16")
    for k in ("q_latent", "q_pe", "kpe_tree", "c_kv", "k_pe"):
        v = inp[k]
        bits = inp[k + "_bits"]
        assert bits.dtype == np.uint16 and bits.shape == v.shape
        assert np.array_equal(v.view(np.uint32) & 0xFFFF, np.zeros(v.shape, np.uint32))
        assert np.array_equal((v.view(np.uint32) >> 16).astype(np.uint16), bits)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20],
                 np.float32)
    got = synth.bf16_to_f32(synth.bf16_bits(x))
    want = np.array([1.0, 1.0, 1.0 + 4 * 2 ** -8, -1.0, 1.0 + 2 * 2 ** -8], np.float32)
    assert np.array_equal(got, want)


def test_deterministic_under_the_seed():
    a, b = synth.generate("cfg4_bf16"), synth.generate("cfg4_bf16")
    for k in ("parent", "prefix_len", "page_table", "q_latent", "c_kv"):
        assert np.array_equal(a[k], b[k])
    c = synth.generate("cfg4_bf16", seed=12345)
    assert not np.array_equal(a["q_latent"], c["q_latent"])


def test_sample_sequences_mixes_chains_and_random_trees():
    inp = synth.generate("cfg5_bf16", DL=8, DR=8, H=1)
    s = synth.sample_sequences(inp, 4)
    assert len(s) == 4 and len(set(s.tolist())) == 4
    assert sum(int(x) % 2 for x in s) == 2                  # two chains, two random trees
    assert np.array_equal(s, synth.sample_sequences(inp, 4))
