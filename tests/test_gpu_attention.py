"""GPU parity: jagged self-attention forward and backward against the fp64 oracle.

Element-by-element comparison on seeded inputs that span several 128-row
tiles with ragged tails (lengths 1, 127, 128, 129, ...), empty sequences,
causal and non-causal masks, head dims 64 / 128 / 192 (192 with the
head-axis chunked backward), the tiny and GEM-like workloads (three sparsity
levels), and the dense causal workload at full size on sampled (sequence,
head) pairs. The longest-first work order is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _gpu(d):
    q, k, v = d["q"].cuda(), d["k"].cuda(), d["v"].cuda()
    off = d["offsets"].cuda()
    return q, k, v, off


def _fwd(d, causal):
    q, k, v, off = _gpu(d)
    o, lse = jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], causal, check=True)
    return o, lse


def _fwd_bwd(d, causal, head_chunk=0):
    q, k, v, off = _gpu(d)
    o, lse = jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], causal, check=True)
    do = d["do"].cuda()
    dq, dk, dv = jfa.jfa_bwd(q, k, v, o, do, lse, off, d["max_seqlen"], d["scale"], causal, head_chunk,
                             check=True)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def _ref_fwd(d, causal):
    return orc.attention_forward(np64(d["q"]), np64(d["k"]), np64(d["v"]), d["offsets"].numpy(), d["scale"], causal)


def _ref_bwd(d, causal):
    return orc.attention_backward(np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), d["offsets"].numpy(),
                                  d["scale"], causal)


def _check_all(d, causal, head_chunk=0, tag=""):
    o, lse, dq, dk, dv = _fwd_bwd(d, causal, head_chunk)
    O_ref, L_ref = _ref_fwd(d, causal)
    check_o(np64(o), O_ref, f"O {tag}")
    check_lse(np64(lse), L_ref, f"LSE {tag}")
    dQ, dK, dV, _ = _ref_bwd(d, causal)
    check_grad(np64(dq), dQ, f"dQ {tag}")
    check_grad(np64(dk), dK, f"dK {tag}")
    check_grad(np64(dv), dV, f"dV {tag}")


def _lengths_case(lengths, heads, head_dim, seed):
    g = torch.Generator().manual_seed(seed)
    return inputs.jagged_from_lengths(torch.tensor(lengths, dtype=torch.int32), heads, head_dim, g)


EDGE = [1, 127, 128, 129, 0, 255, 256, 300, 64, 513]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_config(seed):
    d = inputs.tiny_inputs(seed)
    _check_all(d, False, tag=f"tiny seed {seed}")


@pytest.mark.parametrize("head_dim", [64, 128, 192])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(head_dim, causal):
    d = _lengths_case(EDGE, 2, head_dim, seed=11)
    _check_all(d, causal, tag=f"edges d={head_dim} causal={causal}")


@pytest.mark.parametrize("lengths,head_dim", [([1000], 128), ([256] * 6, 64), ([90] * 5, 192), ([2048], 192)])
@pytest.mark.parametrize("causal", [False, True])
def test_one_sequence_and_equal_lengths(lengths, head_dim, causal):
    """A batch of one sequence (a 16-tile one at head_dim 192 runs the single-stage backward
    through many query tiles, where the TwelveLabs page's deadlock showed) and batches of equal
    lengths, including causal with L < tile."""
    d = _lengths_case(lengths, 1 if lengths[0] == 2048 else 2, head_dim, seed=17)
    _check_all(d, causal, tag=f"lengths {lengths[:2]}.. d={head_dim} causal={causal}")


def test_head_chunk_128_by_64():
    """head_dim 128 run head-axis chunked (two 64-wide slices) equals the unchunked result."""
    d = _lengths_case([200, 77, 129], 2, 128, seed=12)
    _check_all(d, False, head_chunk=64, tag="d=128 chunk 64")


@pytest.mark.parametrize("causal", [False, True])
def test_head_dim_192_three_passes(causal):
    """head_dim 192 with head_chunk 64 (three 64-column passes) instead of the default two
    passes (128 + 64 columns): both must match the oracle."""
    d = _lengths_case([300, 129, 1, 640], 2, 192, seed=18)
    _check_all(d, causal, head_chunk=64, tag=f"d=192 chunk 64 causal={causal}")


@pytest.mark.parametrize("sparsity", [0.1, 0.5, 0.9])
def test_gem_like_reduced_batch(sparsity):
    """GEM-like lengths (max_len 1024, H=4, d=128) on a batch of 24 sequences, full compare."""
    d = inputs.jagged_inputs(24, 1024, sparsity, 4, 128, seed=0)
    _check_all(d, False, tag=f"GEM s={sparsity}")


@pytest.mark.parametrize("sparsity", [0.1, 0.5, 0.9])
def test_gem_like_full_size_sampled(sparsity):
    """The full GEM-like workload (batch 1024) on the GPU; the oracle checks a
    seeded sample of 12 sequences (all heads) element by element."""
    d = inputs.jagged_inputs(1024, 1024, sparsity, 4, 128, seed=0)
    o, lse, dq, dk, dv = _fwd_bwd(d, False)
    o, lse, dq, dk, dv = (np64(t) for t in (o, lse, dq, dk, dv))
    rng = np.random.default_rng(123)
    off = d["offsets"].numpy()
    for b in sorted(rng.choice(1024, 12, replace=False).tolist()):
        s0, s1 = int(off[b]), int(off[b + 1])
        sub = {k: d[k][s0:s1] for k in ("q", "k", "v", "do")}
        one = np.array([0, s1 - s0])
        O_ref, L_ref = orc.attention_forward(np64(sub["q"]), np64(sub["k"]), np64(sub["v"]), one, d["scale"])
        dQ, dK, dV, _ = orc.attention_backward(np64(sub["q"]), np64(sub["k"]), np64(sub["v"]), np64(sub["do"]),
                                               one, d["scale"])
        check_o(o[s0:s1], O_ref, f"O b={b}")
        check_lse(lse[:, s0:s1], L_ref, f"LSE b={b}")
        check_grad(dq[s0:s1], dQ, f"dQ b={b}")
        check_grad(dk[s0:s1], dK, f"dK b={b}")
        check_grad(dv[s0:s1], dV, f"dV b={b}")


@pytest.mark.parametrize("head_dim", [128, 192])
def test_dense_causal_full_size_sampled(head_dim):
    """Batch 4 x 8192 tokens, 16 heads, causal (d=192 with the chunked backward);
    the oracle checks two (sequence, head) pairs in full."""
    d = inputs.dense_causal_inputs(4, 8192, 16, head_dim, seed=0)
    o, lse, dq, dk, dv = _fwd_bwd(d, True)
    o, lse, dq, dk, dv = (np64(t) for t in (o, lse, dq, dk, dv))
    L = 8192
    for b, h in ((0, 0), (3, 11)):
        s0, s1 = b * L, (b + 1) * L
        q, k, v, do = (np64(d[x][s0:s1, h:h + 1]) for x in ("q", "k", "v", "do"))
        one = np.array([0, L])
        O_ref, L_ref = orc.attention_forward(q, k, v, one, d["scale"], True)
        dQ, dK, dV, _ = orc.attention_backward(q, k, v, do, one, d["scale"], True)
        check_o(o[s0:s1, h:h + 1], O_ref, f"O b={b} h={h}")
        check_lse(lse[h:h + 1, s0:s1], L_ref, f"LSE b={b} h={h}")
        check_grad(dq[s0:s1, h:h + 1], dQ, f"dQ b={b} h={h}")
        check_grad(dk[s0:s1, h:h + 1], dK, f"dK b={b} h={h}")
        check_grad(dv[s0:s1, h:h + 1], dV, f"dV b={b} h={h}")


def _queue_from_workspace(ws, batch):
    """Read the work items the queue kernel left in a forward workspace: the
    status block is 256 bytes, the per-sequence tile prefix follows, and the
    items (b, h, t, cost) start at the next 256-byte boundary."""
    raw = ws.cpu()
    n = int(raw[8:12].view(torch.int32)[0])
    start = ((256 + 4 * (batch + 1)) + 255) // 256 * 256
    items = raw[start:start + 16 * n].view(torch.int32).reshape(n, 4).numpy()
    return [(int(b), int(h), int(t)) for b, h, t, _ in items]


@pytest.mark.parametrize("causal", [False, True])
def test_tile_queue_order_bit_exact(causal):
    d = _lengths_case([300, 0, 1, 400, 1000, 129, 128], 3, 64, seed=13)
    q, k, v, off = _gpu(d)
    a_ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], causal, workspace=a_ws, check=True)
    got = _queue_from_workspace(a_ws, len(d["lengths"]))
    assert got == orc.tile_queue(d["offsets"].numpy(), 3, causal, "fwd")


@pytest.mark.parametrize("causal", [False, True])
def test_stream_queue_order_bit_exact(causal):
    """head_dim 128 runs the flat-stream forward; its work items are the same
    longest-first query tiles."""
    d = _lengths_case([300, 0, 1, 400, 1000, 129, 128, 512], 3, 128, seed=16)
    q, k, v, off = _gpu(d)
    a_ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], causal, workspace=a_ws, check=True)
    got = _queue_from_workspace(a_ws, len(d["lengths"]))
    assert got == orc.tile_queue(d["offsets"].numpy(), 3, causal, "fwd")


def test_bad_offsets_are_reported():
    """Offsets inconsistent with the host's total are rejected on the device
    (JFA_ERR_BAD_INPUT) and no work is queued."""
    d = _lengths_case([10, 20], 1, 64, seed=14)
    q, k, v, off = _gpu(d)
    off_bad = off.clone()
    off_bad[1] = 25  # L_1 = -5
    with pytest.raises(jfa.JfaError) as ei:
        jfa.jfa_fwd(q, k, v, off_bad, d["max_seqlen"], d["scale"], False, check=True)
    assert ei.value.status == 6


def test_autograd_wrapper():
    d = _lengths_case([70, 130], 2, 64, seed=15)
    q, k, v, off = _gpu(d)
    q.requires_grad_(True)
    k.requires_grad_(True)
    v.requires_grad_(True)
    o = jfa.jagged_attention(q, k, v, off, d["max_seqlen"], d["scale"])
    o.backward(d["do"].cuda())
    dQ, dK, dV, _ = _ref_bwd(d, False)
    check_grad(np64(q.grad), dQ, "autograd dQ")
    check_grad(np64(k.grad), dK, "autograd dK")
    check_grad(np64(v.grad), dV, "autograd dV")
