"""GPU parity of the causal (prefill) form of tv_verify_attn.

"The Golden Reference: A Pivotal Moment in Building a Native DDTree Inference Engine",
§"Principled Abstraction": one forward_tokens interface serves tree verification,
autoregressive decoding (q_len 1, every key visible) and prefill, the case with causal
masking and no prior cache.  With TV_MASK_CAUSAL query token i (logical key P + i) sees
keys 0 .. P + i, for any q_len.  The oracle computes the same thing as a chain tree (a
chain's ancestor-or-self mask is the causal mask; its depths are 0 .. Q-1, so RoPE puts
token i at P + i as the causal step does with no depth array).
"""
import zlib

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.compare import assert_close, ulp

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def run_prefill(inp, path=tv.PATH_AUTO, num_splits=0, paged_view=tv.PAGED_AUTO):
    assert inp["tree"] == "chain"
    step = VerifyStep(inp, path=path, num_splits=num_splits, paged_view=paged_view, causal=True)
    step.run()
    g = step.results()
    o = oracle.tree_verify_step(inp)
    dt = inp["kv_dtype"]
    assert g["status"] == 0, g["status"]
    assert np.all(np.abs(g["q_pe_rot"] - o["q_pe_rot"]) <= ulp(o["q_pe_rot"], dt))
    assert np.all(np.abs(g["k_pe_cache"] - o["k_pe_cache"]) <= ulp(o["k_pe_cache"], dt))
    e_out = assert_close(g["out"], o["out"], dt, "out", row_len=inp["DL"])
    e_lse = assert_close(g["lse"], o["lse"], dt, "lse", lse=True)
    return step, e_out, e_lse


CASES = [
    # (description, generate kwargs)
    ("prefill 300 tokens, no prior cache, 16 heads", dict(B=1, H=16, Q=300, prefix=(0, 0))),
    ("prefill 257 tokens x 2 sequences, 64 heads", dict(B=2, H=64, Q=257, prefix=(0, 0))),
    ("chunked prefill after a ragged paged prefix",
     dict(B=3, H=16, Q=129, prefix=(100, 700), paged=True)),
    ("prefill 96 tokens, 33 heads (partial tiles)", dict(B=2, H=33, Q=96, prefix=(0, 40))),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("desc,kw", CASES, ids=[c[0] for c in CASES])
def test_prefill_tensor_cores(desc, kw, splits):
    inp = synth.generate(seed=zlib.crc32(desc.encode()) % 1000, dtype="bf16", DL=512, DR=64,
                         tree="chain", **kw)
    step, e_out, e_lse = run_prefill(inp, path=tv.PATH_TCGEN05, num_splits=splits)
    print(desc, splits, e_out["row_rms"], e_lse["scaled"])


@pytest.mark.parametrize("form", [tv.PAGED_STEP_MAPS, tv.PAGED_GATHER],
                         ids=["step-maps", "gathered"])
def test_chunked_prefill_both_paged_forms(form):
    inp = synth.generate(seed=12, dtype="bf16", DL=512, DR=64, tree="chain", B=2, H=64, Q=200,
                         prefix=(500, 1500), paged=True, q_var=0.05)
    run_prefill(inp, path=tv.PATH_TCGEN05, paged_view=form)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("desc,kw", CASES[:3], ids=[c[0] for c in CASES[:3]])
def test_prefill_cuda_cores(desc, kw, dtype):
    kw = dict(kw, DL=512, DR=64)
    inp = synth.generate(seed=zlib.crc32(desc.encode()) % 1000 + 1, dtype=dtype, tree="chain",
                         **kw)
    run_prefill(inp, path=tv.PATH_SIMT)


def test_causal_equals_chain_tree_on_small_q():
    """For q_len <= 64 the causal form and the tree form with a chain tree compute the same
    attention (both within tolerance of the oracle, and of each other)."""
    inp = synth.generate(seed=77, dtype="bf16", DL=512, DR=64, tree="chain", B=3, H=64, Q=33,
                         prefix=(200, 400), paged=True)
    s_tree = VerifyStep(inp, path=tv.PATH_TCGEN05)
    s_tree.run()
    g_tree = s_tree.results()
    step, _, _ = run_prefill(inp, path=tv.PATH_TCGEN05)
    g = step.results()
    assert_close(g["out"], g_tree["out"], "bf16", "causal vs chain tree", row_len=inp["DL"])
    assert np.array_equal(g["q_pe_rot"], g_tree["q_pe_rot"])


def test_tree_mode_still_rejects_long_q():
    inp = synth.generate(seed=5, dtype="bf16", DL=512, DR=64, tree="chain", B=1, H=8, Q=65,
                         prefix=(0, 0))
    step = VerifyStep(inp, causal=True)
    a = step.attn_args()
    a.mask_mode = tv.MASK_TREE
    with pytest.raises(tv.TVError) as e:
        tv.chosen_path(a)
    assert e.value.status == tv.TV_ERR_UNSUPPORTED


def test_full_size_prefill_sampled():
    """The 4096-token, 64-head prefill workload at full size, in the launch configuration
    the benchmark times; sampled tokens checked against the oracle one by one.  Token i of
    a prefill from nothing sees keys 0..i, whose k_pe rows were rotated at their own
    positions: the oracle rebuilds exactly that as a one-node step with a prefix of i keys
    (the prefix rows rotated by the oracle itself)."""
    inp = synth.generate("prefill_bf16")
    step = VerifyStep(inp)
    step.run()
    g = step.results()
    assert g["status"] == 0
    for i in (0, 1, 63, 64, 127, 128, 1000, 2047, 2048, 4094, 4095):
        rot = oracle.rope_neox(inp["kpe_tree"][:, :i, None, :], np.zeros(1, np.int32),
                               np.arange(i, dtype=np.int32)[None, :], inp["rope_base"],
                               out_bf16=True)[0, :, 0, :]
        k_pe = np.zeros((i + 1, inp["DR"]), np.float32)
        k_pe[:i] = rot
        sub = dict(B=1, Q=1, H=inp["H"], DL=inp["DL"], DR=inp["DR"],
                   parent=np.full((1, 1), -1, np.int32),
                   prefix_len=np.full(1, i, np.int32),
                   q_latent=inp["q_latent"][:, i:i + 1], q_pe=inp["q_pe"][:, i:i + 1],
                   kpe_tree=inp["kpe_tree"][:, i:i + 1], c_kv=inp["c_kv"][:i + 1], k_pe=k_pe,
                   page_table=None, page_size=64, kv_stride_b=i + 1, kv_dtype="bf16",
                   q_dtype="bf16", scale=inp["scale"], rope_base=inp["rope_base"])
        o = oracle.tree_verify_step(sub)
        assert_close(g["out"][:, i:i + 1], o["out"], "bf16", f"out token {i}", row_len=inp["DL"])
        assert_close(g["lse"][:, i:i + 1], o["lse"], "bf16", f"lse token {i}", lse=True)
