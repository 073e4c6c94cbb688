"""Bounded waits of the tensor-core attention kernel: make one run out, on purpose and
without any fault, and check that the kernel gives up cleanly.

Every wait of the kernel (on TMA data, on the tensor cores, on the other CTA of its
cluster) has a wall-clock deadline.  The testing hook tv_testing_set_wait_fault stops the
S-side producer of every cluster from issuing key loads and shortens the deadline to
10 ms, so the first wait for a key stage can only end at its deadline.  Expected:
  * the call returns (the stream synchronises) and *status == TV_ERR_TIMEOUT;
  * every CTA of every cluster leaves through the abort path, after its MMAs and copies
    have drained and it has freed its tensor memory (the kernel counts both);
  * a following normal call on the same stream is correct (parity with the oracle), which
    it could not be if tensor memory had been left allocated.
"""
import ctypes

import pytest
import torch

import oracle
from speculative_decoding_tree_04_gb300 import synth, tv
from speculative_decoding_tree_04_gb300.step import VerifyStep
from tests.test_parity_gpu import check_step

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("tvlib")]


@pytest.mark.parametrize("form", [tv.PAGED_STEP_MAPS, tv.PAGED_GATHER],
                         ids=["step-maps", "gathered"])
def test_wait_deadline_aborts_cleanly_and_next_call_is_correct(form):
    inp = synth.generate(seed=404, dtype="bf16", B=2, H=64, Q=9, DL=512, DR=64,
                         prefix=(300, 600), paged=True)
    # one KV split: 2 sequences x 5 row tiles = 10 work items, one per cluster, every one
    # of them with keys to load
    step = VerifyStep(inp, path=tv.PATH_TCGEN05, num_splits=1, paged_view=form)
    step.visibility()
    step.rope_q()
    step.rope_k()
    torch.cuda.synchronize()
    lib = tv.load()
    counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert lib.tv_testing_set_wait_fault(1, 10_000_000, ctypes.c_void_p(counts.data_ptr())) == 0
    try:
        step.attention()
        torch.cuda.synchronize()
    finally:
        assert lib.tv_testing_set_wait_fault(0, 0, None) == 0
    assert int(step.status.item()) == tv.TV_ERR_TIMEOUT
    left, aborted = counts.cpu().tolist()
    assert left == 2 * 10, (left, aborted)      # 10 clusters of 2 CTAs
    assert aborted == left, (left, aborted)     # all of them through the abort path

    # the same stream, the same buffers: a normal call now
    step.status.zero_()
    step.out.fill_(float("nan"))
    step.lse.fill_(float("nan"))
    step.attention()
    g = step.results()
    check_step(inp, g, oracle.tree_verify_step(inp))


def test_hook_rejects_bad_mode():
    assert tv.load().tv_testing_set_wait_fault(2, 0, None) == tv.TV_ERR_INVALID_ARG
