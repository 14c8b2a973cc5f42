"""GPU parity: jagged self-attention forward and backward against the fp64 oracle.

Element-by-element comparison on seeded inputs that span several 128-row
tiles with ragged tails (lengths 1, 127, 128, 129, ...), empty sequences,
causal and non-causal masks, head dims 64 / 128 / 192 (192 with the
head-axis chunked backward), the tiny workload, the GEM-like workload at full
size on every sequence (three sparsity levels; the oracle fans out over the
host cores), and the dense causal workload at full size on 8 seeded (sequence,
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


@pytest.fixture(scope="module")
def oracle_workers():
    """Spawned oracle workers for the full-size checks (one core each)."""
    from tests import oracle_pool
    ex = oracle_pool.pool(mem_per_worker_gb=4.0)
    yield ex
    ex.shutdown()


@pytest.mark.parametrize("sparsity", [0.1, 0.5, 0.9])
def test_gem_like_full_size(sparsity, oracle_workers):
    """The full GEM-like workload (batch 1024, max_len 1024, H 4, d 128) on the
    GPU, every sequence compared with the oracle element by element."""
    from tests import oracle_pool
    d = inputs.jagged_inputs(1024, 1024, sparsity, 4, 128, seed=0)
    gpu = _fwd_bwd(d, False)
    oracle_pool.check_self_full(oracle_workers, d, gpu, False, f"GEM s={sparsity} full")


@pytest.mark.parametrize("head_dim", [128, 192])
def test_dense_causal_full_size_sampled(head_dim, oracle_workers):
    """Batch 4 x 8192 tokens, 16 heads, causal (d=192 with the chunked backward);
    the oracle checks 8 of the 64 (sequence, head) pairs in full, drawn from a
    seeded generator."""
    from tests import oracle_pool
    d = inputs.dense_causal_inputs(4, 8192, 16, head_dim, seed=0)
    gpu = _fwd_bwd(d, True)
    rng = np.random.default_rng(1234 + head_dim)
    pairs = [(int(x) // 16, int(x) % 16) for x in sorted(rng.choice(64, 8, replace=False))]
    oracle_pool.check_self_pairs(oracle_workers, d, gpu, pairs, True, f"dense causal d={head_dim} {pairs}")


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
