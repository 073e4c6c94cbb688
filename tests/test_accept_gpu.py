"""GPU parity of greedy tree acceptance and post-verify compaction (through the C ABI).

tv_tree_accept and tv_compact_kv against the oracle (tree_oracle.c) on the same seeded
inputs: targets, acceptance lengths, paths, emitted tokens and the compacted cache are
integer or byte results and must match bit for bit.  Logits are float32 or bf16 with a
163840-token vocabulary, ties planted at smaller token ids; the trees are the verify
workloads' trees (B8 Q9 and B32 Q33), so the argmax runs with several chunks per row and
with one.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep, _dev_float

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def _dev_logits(acc, dev):
    if acc["logits_dtype"] == "bf16":
        return torch.from_numpy(acc["logits_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(acc["logits"]).to(dev)


def run_accept(inp, acc, dev="cuda"):
    B, Q = inp["B"], inp["Q"]
    logits = _dev_logits(acc, dev)
    parent = torch.from_numpy(inp["parent"]).to(dev)
    tokens = torch.from_numpy(acc["tokens"]).to(dev)
    out = {k: torch.full(shape, -7, dtype=torch.int32, device=dev) for k, shape in
           (("target", (B, Q)), ("accept_len", (B,)), ("path", (B, Q)), ("new_tokens", (B, Q)))}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tv.tree_accept(logits, parent, tokens, out["accept_len"], out["path"], out["new_tokens"],
                   target=out["target"], status=status)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["status"] = int(status.item())
    return res


def check_accept(inp, acc, g):
    tgt = oracle.argmax_rows(acc["logits"])
    a, path, emit = oracle.tree_accept(inp["parent"], acc["tokens"], tgt)
    assert g["status"] == 0
    assert np.array_equal(g["target"], tgt)
    assert np.array_equal(g["accept_len"], a)
    assert np.array_equal(g["path"], path)
    assert np.array_equal(g["new_tokens"], emit)
    return a


@pytest.mark.parametrize("name", ["cfg4_bf16", "cfg5_bf16"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_accept_parity_full_vocabulary(name, dtype):
    inp = synth.generate(name)
    acc = synth.generate_accept(inp, dtype=dtype)
    g = run_accept(inp, acc)
    a = check_accept(inp, acc, g)
    assert a.max() >= 2, a          # the planted paths are taken
    print(name, dtype, "accept lengths", a.tolist())


@pytest.mark.parametrize("V", [1, 5, 13, 2049, 4099])
def test_accept_small_and_ragged_vocabularies(V):
    """Vocabularies that are not whole 16-byte vectors or whole chunks (scalar tail), and
    a single-token vocabulary."""
    inp = synth.generate(seed=31 + V, B=5, H=1, Q=12, DL=8, DR=8, prefix=(1, 1))
    for dtype in ("fp32", "bf16"):
        acc = synth.generate_accept(inp, vocab=V, dtype=dtype, seed=V)
        check_accept(inp, acc, run_accept(inp, acc))


def test_accept_root_only_and_chain():
    inp = synth.generate(seed=3, B=3, H=1, Q=1, DL=8, DR=8, prefix=(1, 1))
    acc = synth.generate_accept(inp, vocab=1000)
    g = run_accept(inp, acc)
    a = check_accept(inp, acc, g)
    assert np.all(a == 0) and np.all(g["new_tokens"][:, 0] == g["target"][:, 0])
    inp = synth.generate(seed=4, B=4, H=1, Q=64, DL=8, DR=8, prefix=(1, 1), tree="chain")
    acc = synth.generate_accept(inp, vocab=3000, p_continue=0.97)
    check_accept(inp, acc, run_accept(inp, acc))


def test_accept_invalid_tree_sets_status():
    inp = synth.generate(seed=5, B=3, H=1, Q=6, DL=8, DR=8, prefix=(1, 1))
    acc = synth.generate_accept(inp, vocab=500)
    inp["parent"][1, 4] = 4
    g = run_accept(inp, acc)
    assert g["status"] == tv.TV_ERR_INVALID_TREE
    assert g["accept_len"][1] == 0 and g["path"][1, 0] == 0 and np.all(g["path"][1, 1:] == -1)
    assert np.all(g["new_tokens"][1] == -1)
    good = [0, 2]
    tgt = oracle.argmax_rows(acc["logits"][good])
    a, path, emit = oracle.tree_accept(inp["parent"][good], acc["tokens"][good], tgt)
    assert np.array_equal(g["accept_len"][good], a) and np.array_equal(g["path"][good], path)


def _cache_arrays(step):
    """The cache as float32 numpy arrays (bf16 caches through their values)."""
    return step.c_kv.float().cpu().numpy(), step.k_pe.float().cpu().numpy()


@pytest.mark.parametrize("name,paged", [("cfg4_bf16", True), ("cfg3_fp32", False),
                                        ("cfg5_bf16", True)])
def test_verify_accept_compact_parity(name, paged):
    """The whole step on the GPU -- visibility, RoPE (the tree k_pe rows go into the cache),
    attention, acceptance, compaction -- against the oracle's same sequence: the compacted
    cache arrays match bit for bit, and so do the new prefix lengths."""
    inp = synth.generate(name)
    if name == "cfg5_bf16":
        inp = synth.generate(name, B=6)
    acc = synth.generate_accept(inp, vocab=32768)
    step = VerifyStep(inp)
    step.run()
    g = run_accept(inp, acc)
    a_dev = torch.from_numpy(g["accept_len"]).cuda()
    p_dev = torch.from_numpy(g["path"]).cuda()
    newp = torch.full((inp["B"],), -1, dtype=torch.int32, device="cuda")
    cache = tv.make_cache(step.page_table, inp["page_size"], inp["kv_stride_b"],
                          min(step.c_kv.shape[0], step.k_pe.shape[0]))
    tv.compact_kv(step.c_kv, step.k_pe, cache, step.prefix_len, p_dev, a_dev, newp,
                  status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    ck, kp = _cache_arrays(step)

    o = oracle.tree_verify_step(inp, seqs=[0])
    a = check_accept(inp, acc, g)
    tgt = oracle.argmax_rows(acc["logits"])
    a, path, _ = oracle.tree_accept(inp["parent"], acc["tokens"], tgt)
    ock, okp, onewp = oracle.compact_kv(inp["c_kv"], o["k_pe_cache"], inp["prefix_len"], path, a,
                                        inp["page_table"], inp["page_size"], inp["kv_stride_b"])
    assert np.array_equal(newp.cpu().numpy(), onewp)
    assert np.array_equal(ck, ock)
    # k_pe: the tree rows were rotated by the GPU and by the oracle separately (within one
    # unit in the last place of the storage format); everything else is moved bytes
    tol = np.spacing(np.abs(okp).astype(np.float32)).astype(np.float64)
    if inp["kv_dtype"] == "bf16":
        tol *= 65536.0
    assert np.all(np.abs(kp - okp) <= tol)
    moved = sum(int((path[b, 1:a[b] + 1] != np.arange(1, a[b] + 1)).sum()) for b in range(inp["B"]))
    print(name, "accepted", a.tolist(), "rows moved", moved)


def test_compaction_rejects_out_of_range_paths():
    inp = synth.generate(seed=9, dtype="bf16", B=2, H=8, Q=9, DL=512, DR=64, prefix=(100, 200),
                         paged=True)
    step = VerifyStep(inp)
    B, Q = inp["B"], inp["Q"]
    path = torch.full((B, Q), -1, dtype=torch.int32, device="cuda")
    path[:, 0] = 0
    path[0, 1] = 3                        # fine
    path[1, 1] = 99                       # outside the tree
    a = torch.tensor([1, 1], dtype=torch.int32, device="cuda")
    newp = torch.zeros(B, dtype=torch.int32, device="cuda")
    before = step.c_kv.clone()
    cache = tv.make_cache(step.page_table, 64, 0, step.c_kv.shape[0])
    tv.compact_kv(step.c_kv, step.k_pe, cache, step.prefix_len, path, a, newp, status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == tv.TV_ERR_BOUNDS
    P = inp["prefix_len"]
    assert newp.cpu().tolist() == [int(P[0]) + 2, int(P[1])]
    # sequence 1 unmoved; sequence 0 moved exactly one row
    diff = (step.c_kv != before).any(dim=1).nonzero().flatten().cpu().tolist()
    pt = inp["page_table"]
    dst = int(pt[0, (P[0] + 1) // 64]) * 64 + (P[0] + 1) % 64
    assert diff in ([dst], [])
