"""The pooled full-size checker on the CPU: it must pass outputs that equal the
oracle rounded to bf16, and catch a planted mistake in any one output of any
one chunk (a flipped dK sign, an O row past its bound, an LSE shift, a wrong
dQ sum), so that a full-size GPU test using it cannot pass vacuously."""
import numpy as np
import pytest
import torch

import oracle.attention as orc
from varlen_flashattention_gb300 import inputs
from tests import oracle_pool
from tests.parity import np64


@pytest.fixture(scope="module")
def ex():
    e = oracle_pool.pool()
    yield e
    e.shutdown()


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


@pytest.fixture(scope="module")
def self_case():
    g = torch.Generator().manual_seed(41)
    d = inputs.jagged_from_lengths(torch.tensor([5, 130, 1, 0, 257, 64], dtype=torch.int32), 2, 64, g)
    off = d["offsets"].numpy()
    O, L = orc.attention_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), off, d["scale"], False)
    dQ, dK, dV, _ = orc.attention_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), off,
                                           d["scale"], False)
    gpu = [_bf16(O), torch.from_numpy(L.astype(np.float32)), _bf16(dQ), _bf16(dK), _bf16(dV)]
    return d, gpu


def test_self_full_passes_exact_outputs(ex, self_case):
    d, gpu = self_case
    oracle_pool.check_self_full(ex, d, gpu, False, "exact", max_rows=100)  # several chunks
    oracle_pool.check_self_pairs(ex, d, gpu, [(1, 0), (4, 1), (2, 1)], False, "pairs")


@pytest.mark.parametrize("which", ["o", "lse", "dk", "dq"])
def test_self_full_catches_a_planted_mistake(ex, self_case, which):
    d, gpu = self_case
    o, lse, dq, dk, dv = (t.clone() for t in gpu)
    s0 = int(d["offsets"][4])  # a row of the fifth sequence (its own chunk)
    if which == "o":
        o[s0 + 3, 1, 7] += 0.05
    elif which == "lse":
        lse[0, s0 + 10] += 2e-3
    elif which == "dk":
        dk[s0:s0 + 257] = -dk[s0:s0 + 257]
    else:
        dq[s0 + 20] *= 1.5
    with pytest.raises(AssertionError):
        oracle_pool.check_self_full(ex, d, (o, lse, dq, dk, dv), False, f"planted {which}", max_rows=100)


def test_bcast_full_checks_every_sequence_and_the_sum(ex):
    d = inputs.broadcast_inputs(batch=5, q_len=40, heads=2, head_dim=64, lk_lo=1, lk_hi=150, seed=42)
    off = d["kv_offsets"].numpy()
    O, L = orc.broadcast_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), off, d["scale"])
    dQ, dK, dV = orc.broadcast_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), off, d["scale"])
    gpu = [_bf16(O), torch.from_numpy(L.astype(np.float32)), _bf16(dQ), _bf16(dK), _bf16(dV)]
    oracle_pool.check_bcast_full(ex, d, gpu, "exact", seqs_per_chunk=2)
    # dQ that misses one sequence's part
    dQ_short = dQ - orc.broadcast_backward(np64(d["q"]), np64(d["k"][off[2]:off[3]]), np64(d["v"][off[2]:off[3]]),
                                           np64(d["do"][2:3]), np.array([0, off[3] - off[2]]), d["scale"])[0]
    with pytest.raises(AssertionError):
        oracle_pool.check_bcast_full(ex, d, [gpu[0], gpu[1], _bf16(dQ_short), gpu[3], gpu[4]], "short dQ",
                                     seqs_per_chunk=2)
    dv_bad = gpu[4].clone()
    dv_bad[int(off[4])] *= -1
    with pytest.raises(AssertionError):
        oracle_pool.check_bcast_full(ex, d, gpu[:4] + [dv_bad], "dV sign", seqs_per_chunk=2)
