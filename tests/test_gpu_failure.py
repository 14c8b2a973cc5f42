"""Failure detection on the GPU, without faulting it.

Every pipeline wait in the library is bounded in time. The self-test kernel
runs that path on purpose: the first stage of a two-stage chain waits for an
input nothing provides, so its wait runs out after a short budget; it must
record JFA_ERR_TIMEOUT with its site code, and the second stage must leave
through the CTA abort flag instead of waiting out its own, longer budget. The
CUDA context must stay usable: a normal call afterwards matches the oracle.
Device-detected bad inputs (offsets, page table) are covered by the parity
test files."""
import time

import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import _abi, inputs
from tests.parity import check_lse, check_o, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("budget_us", [2000, 50000])
def test_wait_timeout_is_reported_and_context_survives(budget_us):
    t0 = time.perf_counter()
    st, detail, aborted = jfa.jfa_selftest_wait_timeout(budget_us)
    elapsed = time.perf_counter() - t0
    assert st == _abi.JFA_ERR_TIMEOUT, st
    assert detail == 901, detail  # the first stage's wait ran out, not the second's
    assert aborted == 1           # the second stage left through the abort flag
    assert elapsed < 5.0 + 8 * budget_us * 1e-6
    # the context is still usable: an ordinary call afterwards is correct
    d = inputs.tiny_inputs(3)
    q, k, v, off = d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), d["offsets"].cuda()
    o, lse = jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], False, check=True)
    O_ref, L_ref = orc.attention_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), d["offsets"].numpy(), d["scale"])
    check_o(np64(o), O_ref, "O after timeout")
    check_lse(np64(lse), L_ref, "LSE after timeout")


def test_status_word_is_reset_by_the_next_call():
    """A call that reuses a workspace clears the previous call's error."""
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    st, _, _ = jfa.jfa_selftest_wait_timeout(2000, workspace=ws)
    assert st == _abi.JFA_ERR_TIMEOUT
    d = inputs.tiny_inputs(4)
    q, k, v, off = d["q"].cuda(), d["k"].cuda(), d["v"].cuda(), d["offsets"].cuda()
    jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], False, workspace=ws)
    assert jfa.jfa_read_device_status(ws) == (_abi.JFA_OK, 0)
