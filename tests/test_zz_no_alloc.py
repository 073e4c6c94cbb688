"""tv_verify_attn_noalloc: the attention for callers that cannot allocate device memory.

Some callers cannot give the library a workspace -- a plugin whose host program owns all
device memory, a serving loop that must not call cudaMalloc/cudaFree (they can stall the
whole device), a fixed memory budget.  For them the split-KV scratch of the CUDA-core
kernel lives in a fixed device array inside the library.  These tests call that entry
point through the C ABI and check it against the regular workspace entry point, twice in
a row with different inputs (the array keeps the previous call's contents, which must
not leak into the next result), and check that an oversized request is refused.

The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.compare import assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


def _both(inp, num_splits):
    step = VerifyStep(inp, path=tv.PATH_SIMT, num_splits=num_splits)
    step.visibility()
    step.rope_q()
    step.rope_k()
    step.attention()                      # regular entry point, torch-provided workspace
    torch.cuda.synchronize()
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    step.out.fill_(float("nan"))
    step.lse.fill_(float("nan"))
    a = step.attn_args()
    assert tv.workspace_size(a) > 0, "this case must use split scratch"
    assert tv.workspace_size(a) <= tv.noalloc_scratch_bytes()
    tv.verify_attn_noalloc(a)             # same arguments, no workspace
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return step, ref_out, ref_lse


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    """Both entry points run the same kernels with the same split plan, so their results
    are identical bit for bit (the tolerance of the parity tests is not needed here)."""
    cases = [(synth.generate("cfg2_fp32", seed=11), 0, "fp32"),
             (synth.generate("cfg3_bf16", seed=12), 3, "bf16")]
    for inp, splits, dt in cases:
        step, ref_out, ref_lse = _both(inp, splits)
        assert torch.equal(step.out, ref_out), "out differs from the workspace entry point"
        assert torch.equal(step.lse, ref_lse), "lse differs from the workspace entry point"
        assert_close(step.out.cpu().numpy(), ref_out.cpu().numpy(), dt, "out")
        assert torch.isfinite(step.out).all() and torch.isfinite(step.lse).all()


def test_noalloc_refuses_requests_beyond_the_fixed_array():
    inp = synth.generate("cfg2_fp32", seed=13)
    step = VerifyStep(inp, path=tv.PATH_SIMT)
    step.visibility()
    a = step.attn_args()
    a.num_splits = 64                     # 33 splits x 544 rows x 513 floats > 32 MiB
    assert tv.workspace_size(a) > tv.noalloc_scratch_bytes()
    with pytest.raises(tv.TVError) as e:
        tv.verify_attn_noalloc(a)
    assert e.value.status == tv.TV_ERR_WORKSPACE
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
