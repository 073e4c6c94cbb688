"""The fused verify prologue (tv_verify_prologue) against the separate calls and the oracle.

One launch does the visibility, the RoPE of the queries' rope part, the RoPE of the draft
keys into their cache slots and the append of the draft tokens' latent rows.  It uses the
separate calls' arithmetic, so its results must equal theirs bit for bit; the latent
rows' cache slots are clobbered first, so the append must write them.  The whole fused
step is then checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.test_parity_gpu import check_step

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def tree_rows(inp):
    B, Q = inp["B"], inp["Q"]
    P = inp["prefix_len"].astype(np.int64)
    jj = P[:, None] + np.arange(Q)[None, :]
    if inp["page_table"] is not None:
        pt = inp["page_table"]
        return pt[np.arange(B)[:, None], jj // 64].astype(np.int64) * 64 + jj % 64
    return np.arange(B)[:, None] * inp["kv_stride_b"] + jj


CASES = [("cfg3_bf16", {}), ("cfg4_bf16", {}), ("cfg1_fp32", {}), ("cfg2_fp32", {}),
         ("cfg5_bf16", dict(B=4))]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_fused_prologue_equals_separate_calls(name, kw):
    inp = synth.generate(name, **kw)
    sep = VerifyStep(inp)
    sep.pre()
    fus = VerifyStep(inp, fused=True)
    rows = torch.from_numpy(tree_rows(inp).ravel()).cuda()
    fus.c_kv[rows] = 0                      # the append must restore these
    fus.k_pe[rows] = 0
    fus.pre()
    torch.cuda.synchronize()
    assert int(fus.status.item()) == 0
    for a, b in ((sep.anc, fus.anc), (sep.depth, fus.depth), (sep.q_pe, fus.q_pe),
                 (sep.k_pe, fus.k_pe), (sep.c_kv, fus.c_kv)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name,kw", [("cfg4_bf16", {}), ("cfg3_fp32", {}),
                                     ("cfg5_bf16", dict(B=3))])
def test_fused_step_parity(name, kw):
    inp = synth.generate(name, **kw)
    step = VerifyStep(inp, fused=True)
    rows = torch.from_numpy(tree_rows(inp).ravel()).cuda()
    step.c_kv[rows] = 0
    step.run()
    check_step(inp, step.results(), oracle.tree_verify_step(inp))


def test_fused_prologue_invalid_tree_and_graph_replay():
    inp = synth.generate(B=3, H=8, Q=6, DL=64, DR=16, prefix=(4, 9), seed=3)
    inp["parent"][1, 3] = 5
    step = VerifyStep(inp, fused=True)
    before = step.q_pe.clone()
    step.pre()
    torch.cuda.synchronize()
    assert int(step.status.item()) == tv.TV_ERR_INVALID_TREE
    assert torch.all(step.depth[1] == -1) and torch.all(step.anc[1] == 0)
    assert torch.equal(step.q_pe[1], before[1])     # the bad sequence is left alone
    # graph replay of the fused step equals the plain call
    inp = synth.generate("cfg4_bf16")
    step = VerifyStep(inp, fused=True)
    step.run()
    ref = step.results()
    g_pre, g_attn = step.capture_graphs()
    for t in (step.out, step.lse, step.q_pe, step.anc, step.depth):
        t.zero_()
    g_pre.replay()
    g_attn.replay()
    got = step.results()
    for k in ("anc", "depth", "q_pe_rot", "k_pe_cache", "out", "lse"):
        assert np.array_equal(got[k], ref[k]), k
    # and so does the whole step as one graph (the preparation overlapping the prologue)
    g_step = step.capture_step_graph()
    for t in (step.out, step.lse, step.q_pe, step.anc, step.depth):
        t.zero_()
    g_step.replay()
    got = step.results()
    for k in ("anc", "depth", "q_pe_rot", "k_pe_cache", "out", "lse"):
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("name,kw", [("cfg4_bf16", {}), ("cfg5_bf16", dict(B=8))])
def test_overlapped_preparation_equals_stream_order(name, kw):
    # tv_attn_args.overlap_prev lets the attention call's preparation run while the
    # prologue finishes; the attention kernel must still see all of the prologue's output.
    # Fresh query inputs on every round, so a stale read would show.
    inp = synth.generate(name, **kw)
    a = VerifyStep(inp, fused=True)
    b = VerifyStep(inp, fused=True)
    gen = torch.Generator(device="cuda").manual_seed(7)
    for _ in range(6):
        fresh = torch.randn(a.q_pe_raw.shape, generator=gen, device="cuda").to(a.q_pe_raw.dtype)
        for st in (a, b):
            st.q_pe_raw.copy_(fresh)
            st.out.zero_()
            st.lse.zero_()
        a.pre()
        a.attention(overlap_prev=False)
        b.run()                                   # overlap_prev = 1
        torch.cuda.synchronize()
        assert int(b.status.item()) == 0
        assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("name,kw,form", [
    ("cfg4_bf16", {}, tv.PAGED_GATHER),          # prep -> key gather -> attention
    ("cfg5_bf16", dict(B=3), tv.PAGED_STEP_MAPS),
    ("cfg2_fp32", {}, tv.PAGED_AUTO),            # CUDA-core path: no preparation kernel
])
def test_overlapped_step_parity_all_forms(name, kw, form):
    """The step with the attention call's preparation overlapping the prologue
    (overlap_prev) against the oracle, for each key view and for the CUDA-core path."""
    inp = synth.generate(name, **kw)
    step = VerifyStep(inp, fused=True, paged_view=form)
    rows = torch.from_numpy(tree_rows(inp).ravel()).cuda()
    step.c_kv[rows] = 0                       # the prologue's append must restore these
    step.run()
    check_step(inp, step.results(), oracle.tree_verify_step(inp))


@pytest.mark.parametrize("name,kw", [("cfg4_bf16", {}), ("cfg3_bf16", {}), ("cfg1_fp32", {})])
def test_host_pipeline_equals_single_steps(name, kw):
    """Steps with host-resident inputs and results, pipelined over two device buffer sets,
    give the results of the same steps run one at a time, bit for bit, and every step
    reads its own inputs (the steps here alternate between two different input sets)."""
    from speculative_decoding_tree_04_gb300.step import HostStepPipeline, _dev_float
    base = synth.generate(name, **kw)
    other = dict(base)  # same sizes, queries negated
    for k in ("q_latent", "q_pe"):
        other[k] = -base[k]
        if base["kv_dtype"] == "bf16":
            other[k + "_bits"] = base[k + "_bits"] ^ np.uint16(0x8000)
    inps = [base, other]
    want = []
    for inp in inps:
        st = VerifyStep(inp, fused=True)
        st.run()
        r = st.results()
        want.append((r["out"], r["lse"]))
    pipe = HostStepPipeline(inps[0], fused=True)
    hosts = []
    for inp in inps:
        h = {k: _dev_float(inp, k, "cuda", pin=True)
             for k in ("q_latent", "q_pe", "kpe_tree", "ckv_tree", "c_kv", "k_pe")}
        h["parent"] = torch.from_numpy(inp["parent"]).pin_memory()
        h["prefix_len"] = torch.from_numpy(inp["prefix_len"]).pin_memory()
        if inp["page_table"] is not None:
            h["page_table"] = torch.from_numpy(inp["page_table"]).pin_memory()
        hosts.append(h)
    shape_o, shape_l = want[0][0].shape, want[0][1].shape
    outs = [(torch.empty(shape_o, dtype=torch.float32).pin_memory(),
             torch.empty(shape_l, dtype=torch.float32).pin_memory()) for _ in range(6)]
    for i in range(6):
        pipe.submit(hosts[i % 2], *outs[i])
    pipe.synchronize()
    for i in range(6):
        o, l = want[i % 2]
        assert np.array_equal(outs[i][0].numpy(), o)
        assert np.array_equal(outs[i][1].numpy(), l)
