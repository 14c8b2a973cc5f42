"""GPU parity past 2^31 elements per tensor: a jagged batch of 8,200 sequences (lengths
U[900, 1148], ~8.4M tokens) with 2 heads of 128 dims, so that Q, K, V, O, dO and the gradients
each hold more than 2^31 elements (~4.3 GB in bf16) and the fp32 dQ accumulator ~8.6 GB: row
and element offsets past the 32-bit range in every kernel (queue, forward, pre-pass, backward,
post-pass), and a batch longer than the queue's shared-memory cache of sequence lengths.

The inputs are drawn on the device (a CPU draw of 2^33 values would dominate the test); the
sequences the oracle checks, in full and element by element, are copied back: the first, two
past the 2^31-element mark and the last.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def test_tensors_past_2_31_elements():
    H, D = 2, 128
    g = torch.Generator().manual_seed(71)
    lengths = inputs.uniform_lengths(8200, 900, 1148, g)
    off = inputs.offsets_from_lengths(lengths)
    T = int(off[-1])
    assert T * H * D > 2 ** 31
    dev = torch.device("cuda", 0)
    q, k, v, do = (inputs.randn_bf16_device((T, H, D), 710 + i, dev) for i in range(4))
    offd = off.to(dev)
    mx, scale = int(lengths.max()), 1.0 / np.sqrt(D)
    o, lse = jfa.jfa_fwd(q, k, v, offd, mx, scale, False, check=True)
    dq, dk, dv = jfa.jfa_bwd(q, k, v, o, do, lse, offd, mx, scale, False, check=True)
    torch.cuda.synchronize()
    first_past = int(np.searchsorted(off.numpy(), 2 ** 31 // (H * D), side="right")) - 1
    for b in sorted({0, first_past, first_past + 1, len(lengths) - 1}):
        s0, s1 = int(off[b]), int(off[b + 1])
        sl = lambda t: np64(t[s0:s1])  # noqa: E731
        sub = np.array([0, s1 - s0])
        O, L = orc.attention_forward(sl(q), sl(k), sl(v), sub, scale, False)
        check_o(sl(o), O, f"O seq {b} (rows {s0}..{s1})")
        check_lse(np64(lse[:, s0:s1]), L, f"LSE seq {b}")
        dQ, dK, dV, _ = orc.attention_backward(sl(q), sl(k), sl(v), sl(do), sub, scale, False)
        check_grad(sl(dq), dQ, f"dQ seq {b}")
        check_grad(sl(dk), dK, f"dK seq {b}")
        check_grad(sl(dv), dV, f"dV seq {b}")


def test_one_long_causal_sequence_sampled_rows():
    """One causal sequence of 65,536 tokens (512 key tiles per head: the queue's longest cost
    buckets, items of up to 512 steps). Sampled query rows are checked one by one: the oracle's
    varlen forward / backward with one query over keys 0..i (bottom-right causal, so it sees all
    of them) gives O, LSE and dQ of that row exactly; dQ is held to 2e-2 of the largest |dQ| of
    the sampled rows (the whole-tensor rule, over the sample)."""
    L, H, D = 65536, 2, 128
    dev = torch.device("cuda", 0)
    q, k, v, do = (inputs.randn_bf16_device((L, H, D), 720 + i, dev) for i in range(4))
    off = torch.tensor([0, L], dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(D)
    o, lse = jfa.jfa_fwd(q, k, v, off, L, scale, True, check=True)
    dq, dk, dv = jfa.jfa_bwd(q, k, v, o, do, lse, off, L, scale, True, check=True)
    torch.cuda.synchronize()
    rows = [0, 127, 128, 40000, 65407, 65535]
    dq_gpu, dq_ref = [], []  # dQ is compared over the whole sample (row 0's exact dQ is 0)
    for i in rows:
        for h in range(H):
            qi, doi = np64(q[i:i + 1, h:h + 1]), np64(do[i:i + 1, h:h + 1])
            K, V = np64(k[:i + 1, h:h + 1]), np64(v[:i + 1, h:h + 1])
            qo, ko = np.array([0, 1]), np.array([0, i + 1])
            O, LS = orc.varlen_forward(qi, K, V, qo, ko, scale, True)
            check_o(np64(o[i:i + 1, h:h + 1]), O, f"O row {i} head {h}")
            check_lse(np64(lse[h:h + 1, i:i + 1]), LS, f"LSE row {i} head {h}")
            dQ, _, _ = orc.varlen_backward(qi, K, V, doi, qo, ko, scale, True)
            dq_gpu.append(np64(dq[i:i + 1, h:h + 1]))
            dq_ref.append(dQ)
    check_grad(np.concatenate(dq_gpu), np.concatenate(dq_ref), f"dQ of rows {rows}")
