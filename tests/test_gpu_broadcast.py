"""GPU parity: broadcast-Q forward and backward (dQ summed over the batch)."""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _run(d):
    q, k, v = d["q"].cuda(), d["k"].cuda(), d["v"].cuda()
    off = d["kv_offsets"].cuda()
    o, lse = jfa.jfa_fwd_broadcast_q(q, k, v, off, d["max_seqlen_k"], d["scale"], check=True)
    dq, dk, dv = jfa.jfa_bwd_broadcast_q(q, k, v, o, d["do"].cuda(), lse, off, d["max_seqlen_k"], d["scale"],
                                         check=True)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("head_dim", [64, 192])
def test_broadcast_head_dims(head_dim):
    """Broadcast-Q at head_dim 64 and 192 (the backward in two head-axis passes)."""
    d = inputs.broadcast_inputs(batch=4, q_len=130, head_dim=head_dim, lk_lo=1, lk_hi=300, seed=2)
    o, lse, dq, dk, dv = _run(d)
    off = d["kv_offsets"].numpy()
    O_ref, L_ref = orc.broadcast_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), off, d["scale"])
    dQ, dK, dV = orc.broadcast_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), off, d["scale"])
    check_o(np64(o), O_ref, f"O d={head_dim}")
    check_lse(np64(lse), L_ref, f"LSE d={head_dim}")
    check_grad(np64(dq), dQ, f"dQ d={head_dim}")
    check_grad(np64(dk), dK, f"dK d={head_dim}")
    check_grad(np64(dv), dV, f"dV d={head_dim}")


@pytest.mark.parametrize("q_len,batch,lo,hi", [(256, 6, 16, 2048), (100, 5, 1, 300), (300, 4, 120, 140)])
def test_broadcast_small(q_len, batch, lo, hi):
    d = inputs.broadcast_inputs(batch=batch, q_len=q_len, lk_lo=lo, lk_hi=hi, seed=1)
    o, lse, dq, dk, dv = _run(d)
    off = d["kv_offsets"].numpy()
    O_ref, L_ref = orc.broadcast_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), off, d["scale"])
    dQ, dK, dV = orc.broadcast_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), off, d["scale"])
    check_o(np64(o), O_ref)
    check_lse(np64(lse), L_ref)
    check_grad(np64(dq), dQ, "dQ (sum over batch)")
    check_grad(np64(dk), dK, "dK")
    check_grad(np64(dv), dV, "dV")


def test_broadcast_full_size():
    """Q [256, 4, 128] shared by 512 jagged K/V sequences (lengths in [16, 2048]):
    O, LSE, dK and dV of every sequence and dQ (the sum over all 512) compared
    with the oracle, which runs in spawned workers over chunks of sequences."""
    from tests import oracle_pool
    d = inputs.broadcast_inputs(seed=0)
    gpu = _run(d)
    ex = oracle_pool.pool(mem_per_worker_gb=2.0)
    try:
        oracle_pool.check_bcast_full(ex, d, gpu, "broadcast-Q full")
    finally:
        ex.shutdown()


def test_broadcast_empty_sequence():
    """A sequence with no keys gets O = 0 and LSE = -inf; its neighbours are unaffected."""
    g = torch.Generator().manual_seed(3)
    lengths = torch.tensor([40, 0, 130], dtype=torch.int32)
    off = inputs.offsets_from_lengths(lengths)
    T = int(off[-1])
    d = {"q": torch.randn(130, 2, 64, generator=g).bfloat16(), "k": torch.randn(T, 2, 64, generator=g).bfloat16(),
         "v": torch.randn(T, 2, 64, generator=g).bfloat16(), "do": torch.randn(3, 130, 2, 64, generator=g).bfloat16(),
         "kv_offsets": off, "max_seqlen_k": 130, "scale": 0.125}
    o, lse, dq, dk, dv = _run(d)
    O_ref, L_ref = orc.broadcast_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), off.numpy(), 0.125)
    dQ, dK, dV = orc.broadcast_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), off.numpy(), 0.125)
    check_o(np64(o), O_ref)
    check_lse(np64(lse), L_ref)
    check_grad(np64(dq), dQ, "dQ")
    check_grad(np64(dk), dK, "dK")
    check_grad(np64(dv), dV, "dV")
