"""Seeded synthetic inputs for tree-verify attention (numpy only, no method arithmetic).

This module draws the raw inputs of one verify step: the draft-tree parent arrays, the
prefix lengths, the absorbed queries, the latent KV cache (contiguous or paged with a
shuffled page pool) and the un-rotated k_pe rows of the draft-tree tokens.  Both the
CUDA path (through the library binding) and the float64 oracle consume these arrays; the
module computes nothing of the method itself (no RoPE, no mask, no softmax).

Workload shapes follow the verify-attention test shapes printed on "The Precision
Imperative: Validating Numerical Accuracy in a Custom CUDA Attention Kernel" (§"The
Message in Full": B/H/q_len/kv_len of each bundle, kv_len = prefix + q_len) and the
absorbed-MLA dimensions d_latent 512 / d_rope 64; value distributions are the synthetic
ones stated with each workload below.  bf16 workloads round every stored value to bf16
(round-to-nearest-even) here, so both sides see identical numbers.
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 64

# name -> workload description.  tree: "random" parent[i] ~ U{0..i-1}; "wide"
# parent[i] ~ U{0..min(i-1,3)}; "mix": odd b chain (parent[i] = i-1), even b random;
# "chain": every sequence a chain; "star": every parent 0.
WORKLOADS = {
    # B3 H8 q_len 5, prefix 1: the smallest printed bundle.
    "cfg1_fp32": dict(B=3, H=8, Q=5, DL=64, DR=16, prefix=(1, 1), tree="random",
                      dtype="fp32", q_var=80.0, scale_den=80.0, paged=False, seed=1001),
    # B2 H16 q_len 17, prefix 2048 (kv_len 2065).
    "cfg2_fp32": dict(B=2, H=16, Q=17, DL=512, DR=64, prefix=(2048, 2048), tree="random",
                      dtype="fp32", q_var=192.0, scale_den=192.0, paged=False, seed=1002),
    # B1 H64 wide tree q_len 33, prefix 128 (kv_len 161), fp32 and bf16 caches.
    "cfg3_fp32": dict(B=1, H=64, Q=33, DL=512, DR=64, prefix=(128, 128), tree="wide",
                      dtype="fp32", q_var=192.0, scale_den=192.0, paged=False, seed=1003),
    "cfg3_bf16": dict(B=1, H=64, Q=33, DL=512, DR=64, prefix=(128, 128), tree="wide",
                      dtype="bf16", q_var=192.0, scale_den=192.0, paged=False, seed=1003),
    # B8 H64 q_len 9, ragged prefix U{1024..4096}, 64-token pages in shuffled order.
    "cfg4_bf16": dict(B=8, H=64, Q=9, DL=512, DR=64, prefix=(1024, 4096), tree="random",
                      dtype="bf16", q_var=192.0, scale_den=192.0, paged=True, seed=1004),
    # B32 H64 q_len 33, chain/random mix, ragged prefix U{4096..8192}, paged, shuffled.
    "cfg5_bf16": dict(B=32, H=64, Q=33, DL=512, DR=64, prefix=(4096, 8192), tree="mix",
                      dtype="bf16", q_var=192.0, scale_den=192.0, paged=True, seed=1005),
    # Prefill of 4096 tokens with no prior cache (the causal form of the same call).
    "prefill_bf16": dict(B=1, H=64, Q=4096, DL=512, DR=64, prefix=(0, 0), tree="chain",
                         dtype="bf16", q_var=192.0, scale_den=192.0, paged=False, seed=1006,
                         causal=True),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _parents(rng, B, Q, tree):
    par = np.zeros((B, Q), np.int32)
    par[:, 0] = -1
    for b in range(B):
        kind = tree
        if tree == "mix":
            kind = "chain" if (b % 2 == 1) else "random"
        for i in range(1, Q):
            if kind == "random":
                par[b, i] = rng.integers(0, i)
            elif kind == "wide":
                par[b, i] = rng.integers(0, min(i - 1, 3) + 1)
            elif kind == "chain":
                par[b, i] = i - 1
            elif kind == "star":
                par[b, i] = 0
            else:
                raise ValueError(kind)
    return par


def generate(name: str | None = None, seed: int | None = None, **kw) -> dict:
    """Draw one verify step's raw inputs.

    ``name`` picks a workload from WORKLOADS; keyword arguments override its fields (B, H,
    Q, DL, DR, prefix=(lo, hi), tree, dtype "fp32"|"bf16", q_var, q_pe_var (rope part of
    the queries; defaults to q_var), scale_den, paged, page size ``page``).  Returns a dict of numpy arrays plus the sizes:

      parent [B,Q] int32, prefix_len [B] int32,
      q_latent [B,Q,H,DL], q_pe [B,Q,H,DR] (un-rotated), kpe_tree [B,Q,DR] (un-rotated),
      ckv_tree [B,Q,DL] (the draft tokens' latent rows, equal to the cache rows at P + i)
      c_kv [rows,DL], k_pe [rows,DR]: the cache (prefix rows and tree latent rows filled,
      every other row finite random data; the tree k_pe rows are written by the verify
      step itself), page_table [B,max_pages] int32 or None, kv_stride_b.

    All float arrays are float32; for bf16 workloads they hold bf16-representable values
    and ``<name>_bits`` (uint16) copies are included for the device.
    """
    cfg = dict(WORKLOADS[name]) if name else {}
    cfg.update(kw)
    cfg.setdefault("page", PAGE)
    cfg.setdefault("q_var", float(cfg["DL"] + cfg["DR"]))
    cfg.setdefault("scale_den", float(cfg["DL"] + cfg["DR"]))
    cfg.setdefault("paged", False)
    cfg.setdefault("tree", "random")
    cfg.setdefault("dtype", "fp32")
    if seed is None:
        seed = cfg.get("seed", 1000)
    B, H, Q, DL, DR = cfg["B"], cfg["H"], cfg["Q"], cfg["DL"], cfg["DR"]
    page = cfg["page"]
    ss = np.random.SeedSequence(seed)
    r_tree, r_pref, r_q, r_qpe, r_ckv, r_kpe, r_kt, r_pages = [
        np.random.default_rng(s) for s in ss.spawn(8)]

    parent = _parents(r_tree, B, Q, cfg["tree"])
    lo, hi = cfg["prefix"]
    prefix_len = r_pref.integers(lo, hi + 1, size=B).astype(np.int32)
    kv_len = prefix_len.astype(np.int64) + Q

    qstd = 1.0 / math.sqrt(cfg["q_var"])
    # q_pe_var (optional) gives the rope part of the queries its own variance 1/q_pe_var
    pstd = 1.0 / math.sqrt(cfg.get("q_pe_var", cfg["q_var"]))
    q_latent = (r_q.standard_normal((B, Q, H, DL), dtype=np.float32) * np.float32(qstd))
    q_pe = (r_qpe.standard_normal((B, Q, H, DR), dtype=np.float32) * np.float32(pstd))
    kpe_tree = r_kt.standard_normal((B, Q, DR), dtype=np.float32)

    if cfg["paged"]:
        npg = (kv_len + page - 1) // page
        max_pages = int(npg.max())
        total = int(npg.sum())
        perm = r_pages.permutation(total).astype(np.int32)
        page_table = np.full((B, max_pages), -1, np.int32)
        off = 0
        for b in range(B):
            page_table[b, : npg[b]] = perm[off: off + npg[b]]
            off += int(npg[b])
        rows = total * page
        kv_stride_b = 0
    else:
        page_table = None
        kv_stride_b = int(((int(kv_len.max()) + page - 1) // page) * page)
        rows = B * kv_stride_b
    c_kv = r_ckv.standard_normal((rows, DL), dtype=np.float32)
    k_pe = r_kpe.standard_normal((rows, DR), dtype=np.float32)

    out = dict(name=name, seed=seed, B=B, H=H, Q=Q, DL=DL, DR=DR, page_size=page,
               kv_stride_b=kv_stride_b, page_table=page_table, parent=parent,
               prefix_len=prefix_len, kv_dtype=cfg["dtype"], q_dtype=cfg["dtype"],
               rope_base=10000.0,
               scale=float(np.float32(1.0 / math.sqrt(cfg["scale_den"]))),
               tree=cfg["tree"], causal=bool(cfg.get("causal", False)))
    # the draft tokens' latent rows (what the step appends into cache slots P + i): the
    # rows the cache holds there
    if cfg["paged"]:
        jj = prefix_len.astype(np.int64)[:, None] + np.arange(Q)[None, :]
        rows_tree = page_table[np.arange(B)[:, None], jj // page].astype(np.int64) * page + jj % page
    else:
        rows_tree = (np.arange(B)[:, None] * kv_stride_b + prefix_len.astype(np.int64)[:, None]
                     + np.arange(Q)[None, :])
    ckv_tree = c_kv[rows_tree]
    arrays = dict(q_latent=q_latent, q_pe=q_pe, kpe_tree=kpe_tree, c_kv=c_kv, k_pe=k_pe,
                  ckv_tree=ckv_tree)
    for k, v in arrays.items():
        if cfg["dtype"] == "bf16":
            bits = bf16_bits(v)
            out[k + "_bits"] = bits
            out[k] = bf16_to_f32(bits)
        else:
            out[k] = np.ascontiguousarray(v, np.float32)
    return out


def sample_sequences(inp: dict, n: int = 4, seed: int = 77) -> np.ndarray:
    """Seeded choice of n sequence indices (half odd, half even when both exist)."""
    rng = np.random.default_rng(seed)
    B = inp["B"]
    if B <= n:
        return np.arange(B, dtype=np.int32)
    odd = np.arange(1, B, 2)
    even = np.arange(0, B, 2)
    k_odd = min(len(odd), n // 2)
    pick = list(rng.choice(odd, k_odd, replace=False)) + \
        list(rng.choice(even, n - k_odd, replace=False))
    return np.sort(np.array(pick, np.int32))



VOCAB = 163840  # vocabulary of the Kimi-K2-class target model the pages build for


def generate_accept(inp: dict, vocab: int = VOCAB, seed: int | None = None,
                    p_continue: float = 0.75, dtype: str = "fp32", ties: bool = True) -> dict:
    """Draft tokens and target logits for greedy tree acceptance over ``inp``'s trees.

    tokens [B,Q] int32: a random token per node, distinct among the children of every
    node unless the vocabulary is smaller than the number of children.  logits [B,Q,vocab] float32 (or bf16-representable values with ``<>_bits``):
    N(0,1) noise, and along one random root path per sequence the logit of the next path
    node's token is raised above the row's maximum (the walk continues there with
    probability p_continue at every step), so that acceptance lengths vary.  With ``ties``
    some rows get their maximum repeated at a smaller token id (the argmax rule must pick
    the smaller).  Numbers only: no acceptance logic is computed here."""
    B, Q = inp["B"], inp["Q"]
    parent = inp["parent"]
    seed = (inp.get("seed", 1000) + 7919) if seed is None else seed
    r_tok, r_log, r_path, r_tie = [np.random.default_rng(s)
                                   for s in np.random.SeedSequence(seed).spawn(4)]
    tokens = np.zeros((B, Q), np.int32)
    for b in range(B):
        tokens[b, 0] = int(r_tok.integers(0, vocab))
        for node in range(Q):
            kids = [c for c in range(1, Q) if parent[b, c] == node]
            if kids:
                # distinct sibling tokens when the vocabulary allows it
                tokens[b, kids] = r_tok.choice(vocab, size=len(kids),
                                               replace=len(kids) > vocab)
    logits = r_log.standard_normal((B, Q, vocab), dtype=np.float32)
    if dtype == "bf16":
        logits = bf16_to_f32(bf16_bits(logits)).reshape(B, Q, vocab)
    for b in range(B):
        cur = 0
        while True:
            kids = [c for c in range(1, Q) if parent[b, c] == cur]
            if not kids or r_path.random() >= p_continue:
                break
            c = int(r_path.choice(kids))
            logits[b, cur, tokens[b, c]] = logits[b, cur].max() + 1.0
            cur = c
    if ties:
        for b in range(B):
            for i in range(Q):
                if r_tie.random() < 0.25:
                    j = int(np.argmax(logits[b, i]))
                    if j > 0:
                        logits[b, i, int(r_tie.integers(0, j))] = logits[b, i, j]
    out = dict(tokens=tokens, logits=logits, vocab=vocab, logits_dtype=dtype)
    if dtype == "bf16":
        # planted values are re-rounded (they stay above the row's other values)
        out["logits_bits"] = bf16_bits(logits)
        out["logits"] = bf16_to_f32(out["logits_bits"]).reshape(B, Q, vocab)
    return out


def generate_draft(B: int, L: int = 16, K: int = 8, vocab: int = VOCAB, seed: int = 2024,
                   concentration: float = 0.7, ties: bool = False) -> dict:
    """Synthetic drafter proposals for best-first tree building: for every sequence and
    depth d = 1..L, K candidate tokens (distinct, random ids) with log-probabilities taken
    from a Dirichlet draw over K + 1 outcomes (the last one stands for the rest of the
    vocabulary), sorted in descending order.  With ``ties`` some neighbouring candidates
    get equal log-probabilities.  Numbers only: no tree is built here."""
    r_p, r_t, r_tie = [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(3)]
    p = r_p.dirichlet(np.full(K + 1, concentration), size=(B, L))[:, :, :K]
    lp = np.log(np.maximum(p, 1e-30)).astype(np.float32)
    lp = -np.sort(-lp, axis=-1)
    if ties:
        m = r_tie.random((B, L, K - 1)) < 0.2 if K > 1 else np.zeros((B, L, 0), bool)
        for k in range(1, K):
            lp[:, :, k] = np.where(m[:, :, k - 1], lp[:, :, k - 1], lp[:, :, k])
    tok = np.stack([np.stack([r_t.choice(vocab, size=K, replace=False) for _ in range(L)])
                    for _ in range(B)]).astype(np.int32)
    root = r_t.integers(0, vocab, size=B).astype(np.int32)
    return dict(logprobs=np.ascontiguousarray(lp), cand_tokens=tok, root=root, L=L, K=K)
