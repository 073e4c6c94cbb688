"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Every test draws seeded synthetic inputs, runs the whole verify step on the GPU
(visibility -> RoPE(q_pe) -> RoPE(tree k_pe into the cache) -> attention) and the same
step in the oracle, and compares:
  * anc bitsets and depths: bit-exact;
  * RoPE outputs: within one unit in the last place of the storage format (device and
    host double-precision cos/sin may differ in the last bit);
  * attention out and lse: max_abs <= 1e-5 and max_rel <= 1e-2 (float32 caches),
    max_abs <= 2e-2 (bf16 caches; the oracle is fed the same bf16 values) together with
    the stricter bf16 rule derived in tests/compare.py (per-row relative rms <= 2^-7 of
    the outputs, lse within 2^-12 relative).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.compare import assert_close, ulp

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def run_pair(inp, path=tv.PATH_AUTO, num_splits=0, seqs=None, paged_view=tv.PAGED_AUTO):
    step = VerifyStep(inp, path=path, num_splits=num_splits, paged_view=paged_view)
    step.run()
    g = step.results()
    o = oracle.tree_verify_step(inp, seqs=seqs)
    return step, g, o


def check_step(inp, g, o, seqs=None):
    dt = inp["kv_dtype"]
    sel = slice(None) if seqs is None else np.asarray(seqs)
    assert g["status"] == 0, tv.load().tv_status_string(g["status"])
    assert np.array_equal(g["anc"], o["anc"])
    assert np.array_equal(g["depth"], o["depth"])
    # RoPE: query rope part and the tree rows written into the cache
    assert np.all(np.abs(g["q_pe_rot"] - o["q_pe_rot"]) <= ulp(o["q_pe_rot"], dt))
    assert np.all(np.abs(g["k_pe_cache"] - o["k_pe_cache"]) <= ulp(o["k_pe_cache"], dt))
    e_out = assert_close(g["out"][sel], o["out"][sel], dt, "out", row_len=inp["DL"])
    e_lse = assert_close(g["lse"][sel], o["lse"][sel], dt, "lse", lse=True)
    return e_out, e_lse


SMALL = ["cfg1_fp32", "cfg2_fp32", "cfg3_fp32", "cfg3_bf16"]


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_workload_parity_simt(name, splits):
    inp = synth.generate(name)
    step, g, o = run_pair(inp, path=tv.PATH_SIMT, num_splits=splits)
    e_out, e_lse = check_step(inp, g, o)
    print(name, "splits", splits, "out", e_out, "lse", e_lse)


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_workload_parity_tc_cfg3(splits):
    inp = synth.generate("cfg3_bf16")
    step, g, o = run_pair(inp, path=tv.PATH_TCGEN05, num_splits=splits)
    print("cfg3 tc splits", splits, check_step(inp, g, o))


@pytest.mark.parametrize("path", [tv.PATH_SIMT, tv.PATH_TCGEN05])
def test_workload_parity_cfg4_both_paths(path):
    inp = synth.generate("cfg4_bf16")
    step, g, o = run_pair(inp, path=path)
    print("cfg4 path", path, check_step(inp, g, o))


def test_auto_path_is_tensor_cores_for_large_bf16():
    for name in ("cfg4_bf16", "cfg5_bf16"):
        inp = synth.generate(name, B=2)
        assert VerifyStep(inp).chosen_path() == tv.PATH_TCGEN05
    assert VerifyStep(synth.generate("cfg2_fp32")).chosen_path() == tv.PATH_SIMT


def test_workload_parity_cfg4_auto():
    inp = synth.generate("cfg4_bf16")
    step, g, o = run_pair(inp)
    print("cfg4 path", step.chosen_path(), check_step(inp, g, o))


@pytest.mark.parametrize("path", [tv.PATH_AUTO, tv.PATH_SIMT])
def test_workload_parity_cfg5_sampled(path):
    inp = synth.generate("cfg5_bf16")
    seqs = synth.sample_sequences(inp, 4)
    step, g, o = run_pair(inp, path=path, seqs=seqs)
    print("cfg5 path", step.chosen_path(), "seqs", seqs, check_step(inp, g, o, seqs=seqs))


def test_cfg5_sharp_softmax_gathered_keys_sampled():
    """The B32 Q33 workload with sharp softmaxes (q_var 0.02: a few keys dominate each row),
    through the per-step maps (automatic) and through the gathered contiguous key view: a
    wrong page or a lost rope term changes the dominant keys and fails the per-row bound by
    orders of magnitude."""
    inp = synth.generate("cfg5_bf16", q_var=0.02)
    seqs = synth.sample_sequences(inp, 4)
    for form in (tv.PAGED_AUTO, tv.PAGED_GATHER):
        step, g, o = run_pair(inp, seqs=seqs, paged_view=form)
        print("cfg5 sharp", form, check_step(inp, g, o, seqs=seqs))


PAGED_FORMS = [tv.PAGED_STEP_MAPS, tv.PAGED_GATHER]
GATHER_CASES = [
    # sharp softmax: frequent rescales, dominant keys
    ("sharp", dict(B=3, H=16, Q=9, prefix=(300, 900), q_var=0.02)),
    # rope-dominant scores: q_latent tiny, q_pe large -- the k_pe of every gathered key
    # (and the rotated tree rows) decides the result
    ("rope-dominant", dict(B=3, H=16, Q=17, prefix=(200, 700), q_var=1e4, q_pe_var=0.05)),
    # 33 heads: the last 128-row tile of a sequence is partial
    ("33 heads", dict(B=2, H=33, Q=5, prefix=(60, 700))),
]


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("form", PAGED_FORMS, ids=["step-maps", "gathered"])
@pytest.mark.parametrize("desc,kw", GATHER_CASES, ids=[c[0] for c in GATHER_CASES])
def test_tc_paged_forms_discriminating(desc, kw, form, splits):
    """Both ways the tensor cores read a paged cache, forced on small caches, against the
    oracle on every sequence."""
    inp = synth.generate(seed=zlib.crc32(desc.encode()) % 1000, dtype="bf16", DL=512, DR=64,
                         paged=True, **kw)
    step, g, o = run_pair(inp, path=tv.PATH_TCGEN05, num_splits=splits, paged_view=form)
    print(desc, form, splits, check_step(inp, g, o))


def test_rope_dominant_scores_simt():
    inp = synth.generate(seed=21, dtype="bf16", B=2, H=16, Q=17, DL=512, DR=64,
                         prefix=(200, 700), q_var=1e4, q_pe_var=0.05, paged=True)
    step, g, o = run_pair(inp, path=tv.PATH_SIMT)
    check_step(inp, g, o)


EDGE = [
    # (description, generate kwargs)
    ("q_len 1 (single-query decode)", dict(B=3, H=8, Q=1, DL=512, DR=64, prefix=(5, 300))),
    ("prefix 0 (pure tree)", dict(B=2, H=8, Q=9, DL=512, DR=64, prefix=(0, 0))),
    ("q_len 64 (bitset limit)", dict(B=2, H=4, Q=64, DL=64, DR=16, prefix=(3, 70))),
    ("kv_len not a multiple of 64, ragged", dict(B=5, H=16, Q=7, DL=128, DR=32, prefix=(1, 200))),
    ("mid-page prefix, paged", dict(B=3, H=16, Q=17, DL=512, DR=64, prefix=(100, 130), paged=True)),
    ("chain trees", dict(B=2, H=8, Q=12, DL=64, DR=16, prefix=(9, 40), tree="chain")),
    ("star trees", dict(B=2, H=8, Q=12, DL=64, DR=16, prefix=(9, 40), tree="star")),
    ("33 heads (partial head group)", dict(B=1, H=33, Q=5, DL=512, DR=64, prefix=(60, 60))),
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("desc,kw", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(desc, kw, dtype):
    inp = synth.generate(seed=zlib.crc32(desc.encode()) % 1000, dtype=dtype, **kw)
    step, g, o = run_pair(inp)
    check_step(inp, g, o)


EDGE_TC = [
    ("tc q_len 1", dict(B=3, H=8, Q=1, prefix=(5, 300))),
    ("tc prefix 0", dict(B=2, H=8, Q=9, prefix=(0, 0))),
    ("tc mid-page prefix, paged", dict(B=3, H=16, Q=17, prefix=(100, 130), paged=True)),
    ("tc 33 heads", dict(B=2, H=33, Q=5, prefix=(60, 700), paged=True)),
    ("tc q_len 64 wide", dict(B=2, H=4, Q=64, prefix=(1, 200), tree="wide")),
    ("tc chain, contiguous", dict(B=2, H=64, Q=12, prefix=(64, 128), tree="chain")),
    ("tc sharp softmax (frequent rescales)", dict(B=2, H=16, Q=9, prefix=(300, 900), q_var=0.02,
                                                  paged=True)),
]


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("desc,kw", EDGE_TC, ids=[e[0] for e in EDGE_TC])
def test_edge_cases_tensor_cores(desc, kw, splits):
    inp = synth.generate(seed=zlib.crc32(desc.encode()) % 1000, dtype="bf16", DL=512, DR=64,
                         **kw)
    step, g, o = run_pair(inp, path=tv.PATH_TCGEN05, num_splits=splits)
    check_step(inp, g, o)


def test_tc_paged_repeated_and_reversed_pages():
    """Paged cache, tensor cores, per-step tensor maps: two logical blocks of one sequence on
    the same physical page (the map's page stride is then zero) and a step whose second page
    lies below its first (the S halves come out swapped).  The oracle reads the same page
    table."""
    inp = synth.generate(seed=77, dtype="bf16", B=2, H=16, Q=5, DL=512, DR=64,
                         prefix=(300, 400), paged=True)
    pt = inp["page_table"].copy()
    pt[0, 1] = pt[0, 0]
    a, b = int(pt[1, 2]), int(pt[1, 3])
    pt[1, 2], pt[1, 3] = max(a, b), min(a, b)
    inp["page_table"] = pt
    step, g, o = run_pair(inp, path=tv.PATH_TCGEN05)
    check_step(inp, g, o)


def test_sharp_softmax_simt():
    inp = synth.generate(seed=5, dtype="fp32", B=2, H=16, Q=9, DL=512, DR=64,
                         prefix=(300, 900), q_var=0.02)
    step, g, o = run_pair(inp, path=tv.PATH_SIMT)
    check_step(inp, g, o)


def test_invalid_tree_sets_status_and_zeroes_that_sequence():
    inp = synth.generate(B=3, H=8, Q=6, DL=64, DR=16, prefix=(4, 9), seed=3)
    inp["parent"][1, 3] = 5  # parent must precede the node
    step = VerifyStep(inp)
    step.run()
    g = step.results()
    assert g["status"] == tv.TV_ERR_INVALID_TREE
    assert np.all(g["anc"][1] == 0) and np.all(g["depth"][1] == -1)
    good = [0, 2]
    o = oracle.tree_verify_step(dict(inp, parent=inp["parent"][good].copy(),
                                     prefix_len=inp["prefix_len"][good].copy(),
                                     q_latent=inp["q_latent"][good], q_pe=inp["q_pe"][good],
                                     kpe_tree=inp["kpe_tree"][good], B=2,
                                     kv_stride_b=inp["kv_stride_b"],
                                     c_kv=np.concatenate([inp["c_kv"][:inp["kv_stride_b"]],
                                                          inp["c_kv"][2 * inp["kv_stride_b"]:]]),
                                     k_pe=np.concatenate([inp["k_pe"][:inp["kv_stride_b"]],
                                                          inp["k_pe"][2 * inp["kv_stride_b"]:]])))
    assert_close(g["out"][good], o["out"], "fp32", "out")
    assert_close(g["lse"][good], o["lse"], "fp32", "lse")
    # the invalid sequence sees only its prefix (no tree key is visible)
    assert np.all(np.isfinite(g["out"][1]))


def test_prefix_beyond_bound_reports_bounds():
    inp = synth.generate(B=2, H=8, Q=5, DL=64, DR=16, prefix=(10, 10), seed=4)
    step = VerifyStep(inp)
    step.max_prefix = 10
    step.prefix_len[1] = 11  # larger than the declared bound
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == tv.TV_ERR_BOUNDS
    assert torch.all(step.out[1] == 0)
    assert torch.all(torch.isinf(step.lse[1]))


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("form", PAGED_FORMS, ids=["step-maps", "gathered"])
def test_guard_bands_untouched_tensor_cores(form, splits):
    """Tensor-core epilogue with a partial last row tile (33 heads x 5 nodes = 165 rows per
    sequence): no store lands outside out / lse, and the results match the oracle."""
    inp = synth.generate(seed=91, dtype="bf16", B=2, H=33, Q=5, DL=512, DR=64,
                         prefix=(60, 700), paged=True)
    step = VerifyStep(inp, path=tv.PATH_TCGEN05, num_splits=splits, paged_view=form)
    B, Q, H, DL = step.B, step.Q, step.H, step.DL
    canary = float.fromhex("0x1.5555p+100")
    big = torch.full((B * Q * H * DL + 2048,), canary, device="cuda")
    step.out = big[1024:1024 + B * Q * H * DL].view(B, Q, H, DL)
    bigl = torch.full((B * Q * H + 2048,), canary, device="cuda")
    step.lse = bigl[1024:1024 + B * Q * H].view(B, Q, H)
    step.run()
    torch.cuda.synchronize()
    assert torch.all(big[:1024] == canary) and torch.all(big[-1024:] == canary)
    assert torch.all(bigl[:1024] == canary) and torch.all(bigl[-1024:] == canary)
    check_step(inp, step.results(), oracle.tree_verify_step(inp))


def test_guard_bands_untouched():
    inp = synth.generate("cfg1_fp32")
    step = VerifyStep(inp)
    B, Q, H, DL = step.B, step.Q, step.H, step.DL
    canary = float.fromhex("0x1.5555p+100")
    big = torch.full((B * Q * H * DL + 2048,), canary, device="cuda")
    step.out = big[1024:1024 + B * Q * H * DL].view(B, Q, H, DL)
    bigl = torch.full((B * Q * H + 2048,), canary, device="cuda")
    step.lse = bigl[1024:1024 + B * Q * H].view(B, Q, H)
    step.run()
    torch.cuda.synchronize()
    assert torch.all(big[:1024] == canary) and torch.all(big[-1024:] == canary)
    assert torch.all(bigl[:1024] == canary) and torch.all(bigl[-1024:] == canary)


def test_q65_unsupported_on_device_call():
    inp = synth.generate(B=1, H=2, Q=8, DL=64, DR=16, prefix=(4, 4), seed=1)
    step = VerifyStep(inp)
    parent = torch.zeros((1, 65), dtype=torch.int32, device="cuda")
    anc = torch.zeros((1, 65), dtype=torch.int64, device="cuda")
    depth = torch.zeros((1, 65), dtype=torch.int32, device="cuda")
    with pytest.raises(tv.TVError) as e:
        tv.build_visibility(parent, anc, depth)
    assert e.value.status == tv.TV_ERR_UNSUPPORTED


def test_dense_mask_matches_oracle():
    inp = synth.generate(B=4, H=1, Q=33, DL=64, DR=16, prefix=(1, 1), seed=8, tree="wide")
    parent = torch.from_numpy(inp["parent"]).cuda()
    anc = torch.empty((4, 33), dtype=torch.int64, device="cuda")
    depth = torch.empty((4, 33), dtype=torch.int32, device="cuda")
    mask = torch.empty((4, 33, 33), dtype=torch.uint8, device="cuda")
    tv.build_visibility(parent, anc, depth, dense_mask=mask)
    vis, dep, ancs = oracle.visibility(inp["parent"])
    assert np.array_equal(mask.cpu().numpy(), vis)
    assert np.array_equal(depth.cpu().numpy(), dep)


def test_all_six_node_trees_bit_exact():
    import itertools
    trees = [np.array([-1, *c], np.int32) for c in itertools.product(*[range(i) for i in range(1, 6)])]
    par = np.stack(trees)
    parent = torch.from_numpy(par).cuda()
    anc = torch.empty(par.shape, dtype=torch.int64, device="cuda")
    depth = torch.empty(par.shape, dtype=torch.int32, device="cuda")
    tv.build_visibility(parent, anc, depth)
    vis, dep, ancs = oracle.visibility(par)
    assert np.array_equal(anc.cpu().numpy().view(np.uint64), ancs)
    assert np.array_equal(depth.cpu().numpy(), dep)


@pytest.mark.parametrize("name", ["cfg3_bf16", "cfg4_bf16"])
def test_graph_replay_matches_plain_calls(name):
    """CUDA-graph replay of the step's calls (as the bench times them) gives the plain calls'
    results bit for bit, and both match the oracle."""
    inp = synth.generate(name)
    step = VerifyStep(inp)
    step.run()
    ref = step.results()
    check_step(inp, ref, oracle.tree_verify_step(inp))
    g_pre, g_attn = step.capture_graphs()
    for t in (step.out, step.lse, step.q_pe, step.anc, step.depth):
        t.zero_()
    for _ in range(2):
        g_pre.replay()
        g_attn.replay()
    got = step.results()
    assert got["status"] == 0
    for k in ("anc", "depth", "q_pe_rot", "k_pe_cache", "out", "lse"):
        assert np.array_equal(got[k], ref[k]), k


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
def test_rope_cancelling_inputs(out_dtype):
    """RoPE on inputs built so that x0*cos - x1*sin (or x1*cos + x0*sin) nearly cancels, or
    sits near 2^-17 .. 2^-21 of |x0*cos| + |x1*sin|: the outputs must still be the float64
    formula rounded once.  Besides one unit in the last place, the bound allows 2^-50 of
    the pair's magnitude, because the device's and libm's double cos/sin may differ in
    their last bit.  Without the exact fallback the error near cancellation is ~2^-44 of
    the magnitude, far above this bound."""
    rng = np.random.default_rng(77)
    B, Q, H, D = 2, 8, 64, 64
    half = D // 2
    P = rng.integers(0, 9000, B).astype(np.int32)
    depth = rng.integers(0, 8, (B, Q)).astype(np.int32)
    pos = (P[:, None] + depth).astype(np.float64)[:, :, None, None]
    inv = 1.0 / np.power(10000.0, 2.0 * np.arange(half) / D)
    c, s = np.cos(pos * inv), np.sin(pos * inv)
    x0 = rng.standard_normal((B, Q, H, half)).astype(np.float32)
    x1 = rng.standard_normal((B, Q, H, half)).astype(np.float32)
    x064 = x0.astype(np.float64)
    mode = np.arange(H)[None, None, :, None] % 4
    ok_s, ok_c = np.abs(s) > 1e-3, np.abs(c) > 1e-3
    a = np.where(ok_s, x064 * c / np.where(ok_s, s, 1.0), x1).astype(np.float32)  # y0 ~ 0
    b = np.where(ok_c, -x064 * s / np.where(ok_c, c, 1.0), x1).astype(np.float32)  # y1 ~ 0
    f = np.exp2(-rng.choice([17.0, 19.0, 21.0], x0.shape))
    t = np.where(ok_s, (x064 * c - f * np.abs(x064 * c)) / np.where(ok_s, s, 1.0), x1)
    x1 = np.where(mode == 0, a, np.where(mode == 1, b, np.where(mode == 2, t.astype(np.float32), x1)))
    x1 = (x1.view(np.int32) + rng.integers(-3, 4, x1.shape).astype(np.int32)).view(np.float32)
    x = np.concatenate([x0, x1], axis=-1).astype(np.float32)

    dev = torch.device("cuda")
    xt = torch.from_numpy(x).to(dev)
    out = torch.empty(x.shape, dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16,
                      device=dev)
    tv.rope_neox(xt, out, torch.from_numpy(P).to(dev), torch.from_numpy(depth).to(dev))
    g = out.float().cpu().numpy()
    o = oracle.rope_neox(x, P, depth, out_bf16=(out_dtype == "bf16"))
    mag = np.abs(x[..., :half]) + np.abs(x[..., half:])
    bound = ulp(o, out_dtype) + np.exp2(-50.0) * np.concatenate([mag, mag], axis=-1)
    assert np.all(np.abs(g - o) <= bound), float(np.max(np.abs(g - o) / bound))


@pytest.mark.parametrize("in_dt,out_dt", [(torch.float32, torch.float32),
                                          (torch.bfloat16, torch.bfloat16),
                                          (torch.float32, torch.bfloat16)])
def test_rope_vector_and_elementwise_forms_agree(in_dt, out_dt):
    """tv_rope_neox takes a vector form (four rotate-half pairs per load) when d_rope is a
    multiple of 8 and the strides are multiples of four elements, and an element-wise form
    otherwise; both use the same arithmetic, so their results must be the same bits."""
    torch.manual_seed(5)
    dev = torch.device("cuda")
    B, Q, H, D = 3, 9, 64, 64
    P = torch.randint(0, 5000, (B,), dtype=torch.int32, device=dev)
    depth = torch.randint(0, Q, (B, Q), dtype=torch.int32, device=dev)
    x = torch.randn(B, Q, H, D, device=dev).to(in_dt)
    wide = torch.zeros(B, Q, H, D + 2, device=dev, dtype=in_dt)
    wide[..., :D] = x
    xs = wide[..., :D]                       # head stride D + 2: the element-wise form
    ov = torch.empty(B, Q, H, D, device=dev, dtype=out_dt)
    os_ = torch.empty_like(ov)
    tv.rope_neox(x, ov, P, depth)
    tv.rope_neox(xs, os_, P, depth)
    torch.cuda.synchronize()
    assert torch.equal(ov, os_)


@pytest.mark.parametrize("in_dt", [torch.float32, torch.bfloat16])
def test_rope_bf16_store_equals_rounded_float32_result(in_dt):
    """For bf16 storage the rotation first tries plain float32 arithmetic and keeps it when
    the bf16 rounding is already decided; otherwise it takes the exact path.  The stored
    bits must equal the float32 result (the exact path) rounded to bf16, also for inputs
    built to cancel."""
    rng = np.random.default_rng(11)
    dev = torch.device("cuda")
    B, Q, H, D = 2, 8, 64, 64
    half = D // 2
    P = rng.integers(0, 9000, B).astype(np.int32)
    depth = rng.integers(0, 8, (B, Q)).astype(np.int32)
    pos = (P[:, None] + depth).astype(np.float64)[:, :, None, None]
    inv = 1.0 / np.power(10000.0, 2.0 * np.arange(half) / D)
    c, s = np.cos(pos * inv), np.sin(pos * inv)
    x0 = rng.standard_normal((B, Q, H, half)).astype(np.float32)
    x1 = rng.standard_normal((B, Q, H, half)).astype(np.float32)
    ok = np.abs(s) > 1e-3
    near = np.where(ok, x0.astype(np.float64) * c / np.where(ok, s, 1.0), x1).astype(np.float32)
    x1 = np.where((np.arange(H) % 2 == 0)[None, None, :, None], near, x1)
    x1 = (x1.view(np.int32) + rng.integers(-2, 3, x1.shape).astype(np.int32)).view(np.float32)
    x = torch.from_numpy(np.concatenate([x0, x1], axis=-1)).to(dev).to(in_dt)
    Pt, dt = torch.from_numpy(P).to(dev), torch.from_numpy(depth).to(dev)
    o32 = torch.empty(B, Q, H, D, device=dev, dtype=torch.float32)
    o16 = torch.empty(B, Q, H, D, device=dev, dtype=torch.bfloat16)
    tv.rope_neox(x, o32, Pt, dt)
    tv.rope_neox(x, o16, Pt, dt)
    torch.cuda.synchronize()
    assert torch.equal(o16, o32.to(torch.bfloat16))


@pytest.mark.parametrize("B,lo,hi", [(2, 1500, 3000), (9, 2000, 2600), (76, 1, 600),
                                      (80, 1, 300)])
def test_schedule_shapes_tensor_cores(B, lo, hi):
    """Batch sizes whose row tiles (17 per sequence at q_len 33, 64 heads) fall below, just
    past, exactly on and past a whole number of rounds over the 76 clusters of a GB300: every
    tile split in pieces; two rounds and one tile split; whole rounds only; 68 tiles left
    over, one piece each.  Ragged prefixes in a paged cache, every sequence against the
    oracle."""
    inp = synth.generate("cfg5_bf16", B=B, prefix=(lo, hi), seed=500 + B)
    step, g, o = run_pair(inp, path=tv.PATH_TCGEN05)
    check_step(inp, g, o)


@pytest.mark.parametrize("name,kw", [("cfg4_bf16", {}), ("cfg5_bf16", dict(B=4))])
def test_repeated_calls_bit_identical(name, kw):
    """The tensor-core call is deterministic: the schedule depends only on the sizes and
    prefix lengths, and every sum (softmax, P.V, the merge of split tiles) runs in a fixed
    order, so a second call gives the same bits."""
    inp = synth.generate(name, **kw)
    step = VerifyStep(inp, path=tv.PATH_TCGEN05)
    step.run()
    first = step.results()
    for _ in range(2):
        step.attention()
        again = step.results()
        assert np.array_equal(again["out"], first["out"])
        assert np.array_equal(again["lse"], first["lse"])
