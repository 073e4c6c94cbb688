"""One tree-verify step on the GPU, composed from the library's three calls.

``VerifyStep`` holds the device buffers of a step (draft-tree parents, prefix lengths,
queries, the latent KV cache, outputs) and runs, on one CUDA stream:

    tv_build_visibility(parent)                     -> anc, depth
    tv_rope_neox(q_pe, in place, pos = P + depth)   -> rotated query rope part
    tv_rope_neox(kpe_tree -> cache rows P + i)      -> rotated draft-token k_pe in cache
    tv_verify_attn(...)                             -> out [B,Q,H,DL], lse [B,Q,H]

``HostStepPipeline`` runs steps whose inputs and results live in host memory, with each
step's copies overlapping its neighbours' work.

This module moves bytes and issues calls; all arithmetic runs in libtv's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import tv


def _dev_float(inp: dict, key: str, device, pin=False):
    if inp["kv_dtype"] == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(inp[key + "_bits"]).view(np.int16)).view(
            torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(inp[key], np.float32))
    if pin:
        return t.pin_memory()
    return t.to(device)


class VerifyStep:
    """Device-resident inputs/outputs of one verify step plus the call sequence."""

    HOST_KEYS = ("parent", "prefix_len", "page_table", "q_latent", "q_pe", "kpe_tree",
                 "c_kv", "k_pe")

    def __init__(self, inp: dict, device="cuda", path=tv.PATH_AUTO, num_splits=0,
                 paged_view=tv.PAGED_AUTO, causal=None, fused=False):
        self.inp = inp
        self.device = torch.device(device)
        self.path = path
        self.num_splits = num_splits
        self.paged_view = paged_view
        # causal: prefill of Q tokens after the prefix (no draft tree: no visibility call,
        # token i at position P + i, the causal mask); by default the workload's own mode
        self.causal = bool(inp.get("causal", False)) if causal is None else causal
        self.mask_mode = tv.MASK_CAUSAL if self.causal else tv.MASK_TREE
        # fused: visibility, both RoPE calls and the append of the draft latent rows as one
        # tv_verify_prologue launch (tree steps only)
        self.fused = bool(fused) and not self.causal
        d = self.device
        B, Q, H, DL = inp["B"], inp["Q"], inp["H"], inp["DL"]
        self.B, self.Q, self.H, self.DL, self.DR = B, Q, H, DL, inp["DR"]
        self.parent = torch.from_numpy(inp["parent"]).to(d)
        self.prefix_len = torch.from_numpy(inp["prefix_len"]).to(d)
        self.page_table = (None if inp["page_table"] is None
                           else torch.from_numpy(inp["page_table"]).to(d))
        self.q_latent = _dev_float(inp, "q_latent", d)
        self.q_pe_raw = _dev_float(inp, "q_pe", d)
        self.kpe_tree = _dev_float(inp, "kpe_tree", d)
        self.ckv_tree = _dev_float(inp, "ckv_tree", d)
        self.c_kv = _dev_float(inp, "c_kv", d)
        self.k_pe = _dev_float(inp, "k_pe", d)
        self.q_pe = torch.zeros_like(self.q_pe_raw)
        self.anc = None if self.causal else torch.empty((B, Q), dtype=torch.int64, device=d)
        self.depth = None if self.causal else torch.empty((B, Q), dtype=torch.int32, device=d)
        self.out = torch.empty((B, Q, H, DL), dtype=torch.float32, device=d)
        self.lse = torch.empty((B, Q, H), dtype=torch.float32, device=d)
        self.status = torch.zeros(1, dtype=torch.int32, device=d)
        self.max_prefix = int(inp["prefix_len"].max()) if B else 0
        self.cache = tv.make_cache(self.page_table, inp["page_size"], inp["kv_stride_b"],
                                   min(self.c_kv.shape[0], self.k_pe.shape[0]))
        self.workspace = None
        self._alloc_workspace()

    def attn_args(self):
        return tv.attn_args(self.q_latent, self.q_pe, self.c_kv, self.k_pe, self.prefix_len,
                            self.anc, self.out, self.lse, self.inp["scale"], self.max_prefix,
                            self.page_table, self.inp["page_size"], self.inp["kv_stride_b"],
                            self.status, self.path, self.num_splits, self.paged_view,
                            self.mask_mode)

    def _alloc_workspace(self):
        need = tv.workspace_size(self.attn_args())
        self.workspace = (torch.empty(need, dtype=torch.uint8, device=self.device)
                          if need > 0 else None)

    def chosen_path(self) -> int:
        return tv.chosen_path(self.attn_args())

    # -- the four calls of one step ------------------------------------------------
    def visibility(self, stream=None):
        if self.causal:
            return  # no tree to resolve
        tv.build_visibility(self.parent, self.anc, self.depth, status=self.status,
                            stream=stream)

    def rope_q(self, stream=None):
        tv.rope_neox(self.q_pe_raw, self.q_pe, self.prefix_len, self.depth,
                     self.inp["rope_base"], stream=stream)

    def rope_k(self, stream=None):
        tv.rope_neox(self.kpe_tree, self.k_pe, self.prefix_len, self.depth,
                     self.inp["rope_base"], cache=self.cache, stream=stream)

    def attention(self, stream=None, overlap_prev=False):
        """The attention call.  overlap_prev: the work queued just before it is this step's
        prologue, which writes neither prefix_len nor the page table, so the call's
        preparation may overlap it (tv_attn_args.overlap_prev)."""
        tv.verify_attn(self.q_latent, self.q_pe, self.c_kv, self.k_pe, self.prefix_len,
                       self.anc, self.out, self.lse, self.inp["scale"], self.max_prefix,
                       self.page_table, self.inp["page_size"], self.inp["kv_stride_b"],
                       self.status, self.path, self.num_splits, workspace=self.workspace,
                       stream=stream, paged_view=self.paged_view, mask_mode=self.mask_mode,
                       overlap_prev=1 if overlap_prev else 0)

    def prologue(self, stream=None):
        tv.verify_prologue(self.parent, self.prefix_len, self.q_pe_raw, self.q_pe,
                           self.kpe_tree, self.ckv_tree, self.c_kv, self.k_pe, self.cache,
                           self.anc, self.depth, self.inp["rope_base"], status=self.status,
                           stream=stream)

    def pre(self, stream=None):
        """Everything before the attention: one fused launch, or the separate calls."""
        if self.fused:
            self.prologue(stream)
        else:
            self.visibility(stream)
            self.rope_q(stream)
            self.rope_k(stream)

    def run(self, stream=None):
        self.pre(stream)
        self.attention(stream, overlap_prev=self.fused)

    def capture_graphs(self):
        """Capture the step as two CUDA graphs: (visibility, both RoPE calls) and the
        attention call.  Replaying them launches the same kernels with the same arguments as
        ``run()`` without the host's per-call work.  The calls run once eagerly first, so
        that the library's one-time set-up (occupancy query, driver entry points) happens
        outside the capture.  The graphs keep this step's buffers and sizes."""
        cur = torch.cuda.current_stream(self.device)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            self.run()
        cur.wait_stream(side)
        torch.cuda.synchronize(self.device)
        g_pre, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre):
            self.pre()
        with torch.cuda.graph(g_attn):
            self.attention()
        return g_pre, g_attn

    def capture_step_graph(self):
        """Capture the whole step (the calls before attention, then the attention call) as
        one CUDA graph: one launch per step instead of two.  Call after ``capture_graphs``
        (or ``run``), which does the library's one-time set-up outside any capture."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.pre()
            self.attention(overlap_prev=self.fused)
        return g

    def launches_per_step(self) -> int:
        """Kernels one run() enqueues: visibility (not for causal prefill) and 2 RoPE, or
        the fused prologue, and the attention call's own."""
        pre = 1 if self.fused else (2 if self.causal else 3)
        return pre + tv.attn_launches(self.attn_args())

    # -- results --------------------------------------------------------------------
    def results(self):
        torch.cuda.synchronize(self.device)
        anc = None if self.anc is None else self.anc.cpu().numpy().view(np.uint64)
        return dict(anc=anc, depth=None if self.depth is None else self.depth.cpu().numpy(),
                    q_pe_rot=self.q_pe.float().cpu().numpy(),
                    k_pe_cache=self.k_pe.float().cpu().numpy(),
                    out=self.out.cpu().numpy(), lse=self.lse.cpu().numpy(),
                    status=int(self.status.item()))


class HostStepPipeline:
    """Verify steps whose inputs and results live in host memory, pipelined on the GPU.

    Two device buffer sets (two ``VerifyStep``) and three CUDA streams: step i uploads its
    inputs (pinned host tensors, keyed like ``VerifyStep.HOST_KEYS``) into buffer set i % 2
    on the upload stream, runs on the compute stream once its upload is done, and
    downloads out and lse into the host tensors given for it on the download stream once
    it has run.  So step i + 1's upload overlaps step i's compute and step i's download,
    and a buffer set is reused only after its previous download has finished.  Every step
    still copies all of its inputs in and its results out.  ``synchronize()`` waits for all
    submitted steps; results must not be read, nor a step's host inputs changed, before
    it (the copies run asynchronously from pinned memory)."""

    def __init__(self, inp: dict, device="cuda", **step_kw):
        self.device = torch.device(device)
        self.steps = [VerifyStep(inp, device=self.device, **step_kw) for _ in range(2)]
        self.streams = [torch.cuda.Stream(self.device) for _ in range(3)]
        self._done = [None, None]
        self._n = 0

    def _dst(self, st: "VerifyStep") -> dict:
        return {"q_latent": st.q_latent, "q_pe": st.q_pe_raw, "kpe_tree": st.kpe_tree,
                "ckv_tree": st.ckv_tree, "c_kv": st.c_kv, "k_pe": st.k_pe,
                "parent": st.parent, "prefix_len": st.prefix_len, "page_table": st.page_table}

    def submit(self, host_in: dict, out_h: torch.Tensor, lse_h: torch.Tensor):
        """Queue one step: copy ``host_in`` (name -> pinned tensor) in, run, copy out and
        lse into the pinned ``out_h`` and ``lse_h``.  Returns at once."""
        b = self._n % 2
        self._n += 1
        st = self.steps[b]
        dst = self._dst(st)
        s_in, s_c, s_out = self.streams
        start = torch.cuda.Event()
        start.record(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s_in):
            s_in.wait_event(start)
            if self._done[b] is not None:
                s_in.wait_event(self._done[b])
            for k, t in host_in.items():
                dst[k].copy_(t, non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(e_in)
            st.run(s_c)
            e_c = torch.cuda.Event()
            e_c.record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_c)
            out_h.copy_(st.out, non_blocking=True)
            lse_h.copy_(st.lse, non_blocking=True)
            e_o = torch.cuda.Event()
            e_o.record(s_out)
            self._done[b] = e_o

    def wait_on(self, stream=None):
        """Make ``stream`` (default: the current one) wait for every submitted step."""
        cur = stream if stream is not None else torch.cuda.current_stream(self.device)
        for s in self.streams:
            cur.wait_stream(s)

    def synchronize(self):
        for s in self.streams:
            s.synchronize()
