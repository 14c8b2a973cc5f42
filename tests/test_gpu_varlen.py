"""GPU parity: varlen attention (separate query / key lengths, grouped KV heads).

Element-by-element comparison with the fp64 oracle on seeded inputs: query
and key lengths that differ per sequence (ragged tails around 128-row tiles,
empty query or key sides, L_q > L_k with the bottom-right causal mask leaving
rows that see no key), GQA group sizes 1 / 4 and MQA, head dims 64 / 128 /
192, causal and not. The longest-first work order of both passes is compared
bit for bit with the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _case(q_lengths, k_lengths, q_heads, kv_heads, head_dim, seed):
    g = torch.Generator().manual_seed(seed)
    return inputs.varlen_from_lengths(q_lengths, k_lengths, q_heads, kv_heads, head_dim, g)


def _run(d, causal, ws_f=None, ws_b=None):
    q, k, v, do = (d[x].cuda() for x in ("q", "k", "v", "do"))
    qo, ko = d["q_offsets"].cuda(), d["k_offsets"].cuda()
    o, lse = jfa.jfa_fwd_varlen(q, k, v, qo, ko, d["max_seqlen_q"], d["max_seqlen_k"], d["scale"], causal,
                                workspace=ws_f, check=True)
    dq, dk, dv = jfa.jfa_bwd_varlen(q, k, v, o, do, lse, qo, ko, d["max_seqlen_q"], d["max_seqlen_k"], d["scale"],
                                    causal, workspace=ws_b, check=True)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def _check(d, causal, tag):
    o, lse, dq, dk, dv = _run(d, causal)
    args = (np64(d["q"]), np64(d["k"]), np64(d["v"]))
    qo, ko = d["q_offsets"].numpy(), d["k_offsets"].numpy()
    O_ref, L_ref = orc.varlen_forward(*args, qo, ko, d["scale"], causal)
    check_o(np64(o), O_ref, f"O {tag}")
    check_lse(np64(lse), L_ref, f"LSE {tag}")
    dQ, dK, dV = orc.varlen_backward(*args, np64(d["do"]), qo, ko, d["scale"], causal)
    check_grad(np64(dq), dQ, f"dQ {tag}")
    check_grad(np64(dk), dK, f"dK {tag}")
    check_grad(np64(dv), dV, f"dV {tag}")
    return O_ref, L_ref


# (L_q, L_k) pairs: ragged tails, L_q < L_k (chunked prefill), L_q > L_k
# (rows with no visible key under the bottom-right mask), empty sides, L_q = 1
Q_LENS = [130, 1, 300, 0, 129, 40, 256, 200, 5]
K_LENS = [500, 700, 129, 64, 0, 300, 256, 77, 5]


@pytest.mark.parametrize("head_dim", [64, 128, 192])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_gqa(head_dim, causal):
    d = _case(Q_LENS, K_LENS, 8, 2, head_dim, seed=31)
    O_ref, L_ref = _check(d, causal, f"gqa d={head_dim} causal={causal}")
    if causal:  # sequence 2 (query rows 131 .., L_q 300, L_k 129): its first 171 rows see no key
        assert np.isneginf(L_ref[:, 131:131 + 171]).all() and np.isfinite(L_ref[:, 131 + 171]).all()


@pytest.mark.parametrize("kv_heads", [1, 4])
def test_varlen_mqa_and_mha(kv_heads):
    d = _case([257, 64, 1000], [128, 900, 1000], 4, kv_heads, 128, seed=32)
    _check(d, True, f"Hkv={kv_heads}")


def test_varlen_self_equals_jfa_fwd():
    """Equal query and key packing with one KV head per query head is jagged
    self-attention: the varlen entry points agree with jfa_fwd / jfa_bwd."""
    d = _case([300, 17, 128], [300, 17, 128], 2, 2, 128, seed=33)
    o, lse, dq, dk, dv = _run(d, True)
    q, k, v, do = (d[x].cuda() for x in ("q", "k", "v", "do"))
    off = d["q_offsets"].cuda()
    o2, lse2 = jfa.jfa_fwd(q, k, v, off, 300, d["scale"], True, check=True)
    dq2, dk2, dv2 = jfa.jfa_bwd(q, k, v, o2, do, lse2, off, 300, d["scale"], True, check=True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    check_grad(np64(dq), np64(dq2), "dQ varlen vs self")  # dQ sums in nondeterministic order


def test_varlen_reduced_gem_like():
    """Jagged GQA batch at the GEM-like scale of lengths (U[1, 1024] on both
    sides, 8 query heads on 2 KV heads, head_dim 128), 16 sequences."""
    d = inputs.varlen_inputs(16, 1, 1024, 1, 1024, 8, 2, 128, seed=34)
    _check(d, True, "gem-like varlen causal")


def _items(ws, batch, n_index=2):
    raw = ws.cpu()
    n = int(raw[4 * n_index:4 * n_index + 4].view(torch.int32)[0])
    start = ((256 + 4 * (batch + 1)) + 255) // 256 * 256
    items = raw[start:start + 16 * n].view(torch.int32).reshape(n, 4).numpy()
    return [(int(b), int(h), int(t)) for b, h, t, _ in items]


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_queue_order_bit_exact(causal):
    d = _case([300, 0, 1, 700, 1000, 129, 100], [100, 400, 300, 0, 1300, 50, 1000], 4, 2, 64, seed=35)
    ws_f = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    ws_b = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")
    _run(d, causal, ws_f, ws_b)
    B = len(d["q_lengths"])
    qo, ko = d["q_offsets"].numpy(), d["k_offsets"].numpy()
    assert _items(ws_f, B) == orc.varlen_tile_queue(qo, ko, 4, 2, causal, "fwd")
    assert _items(ws_b, B) == orc.varlen_tile_queue(qo, ko, 4, 2, causal, "bwd")


def test_varlen_bad_key_offsets_are_reported():
    d = _case([10, 20], [30, 5], 2, 1, 64, seed=36)
    q, k, v = (d[x].cuda() for x in ("q", "k", "v"))
    qo, ko = d["q_offsets"].cuda(), d["k_offsets"].cuda()
    ko_bad = ko.clone()
    ko_bad[1] = 40  # L_k of sequence 1 becomes -5
    with pytest.raises(jfa.JfaError) as ei:
        jfa.jfa_fwd_varlen(q, k, v, qo, ko_bad, 20, 30, d["scale"], False, check=True)
    assert ei.value.status == 6


def test_varlen_autograd_wrapper():
    d = _case([70, 130], [200, 30], 4, 2, 64, seed=37)
    q, k, v = (d[x].cuda().requires_grad_(True) for x in ("q", "k", "v"))
    qo, ko = d["q_offsets"].cuda(), d["k_offsets"].cuda()
    o = jfa.varlen_attention(q, k, v, qo, ko, 130, 200, d["scale"], True)
    o.backward(d["do"].cuda())
    args = (np64(d["q"]), np64(d["k"]), np64(d["v"]), np64(d["do"]), d["q_offsets"].numpy(), d["k_offsets"].numpy())
    dQ, dK, dV = orc.varlen_backward(*args, d["scale"], True)
    check_grad(np64(q.grad), dQ, "autograd dQ")
    check_grad(np64(k.grad), dK, "autograd dK")
    check_grad(np64(v.grad), dV, "autograd dV")


def test_varlen_prefill_full_size_sampled():
    """The chunked-prefill workload the bench times (64 sequences, L_q U[1, 1024] at the end of
    L_k = L_q + U[0, 3072] keys, 32 query heads on 8 KV heads, d 128, causal) at full size; the
    oracle checks forward and backward of three sampled sequences."""
    g = torch.Generator().manual_seed(38)
    ql = inputs.uniform_lengths(64, 1, 1024, g)
    kl = ql + inputs.uniform_lengths(64, 0, 3072, g)
    d = inputs.varlen_from_lengths(ql, kl, 32, 8, 128, g)
    o, lse, dq, dk, dv = _run(d, True)
    qo, ko = d["q_offsets"].numpy(), d["k_offsets"].numpy()
    for b in (0, 31, 63):
        q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
        one_q, one_k = np.array([0, q1 - q0]), np.array([0, k1 - k0])
        args = (np64(d["q"][q0:q1]), np64(d["k"][k0:k1]), np64(d["v"][k0:k1]))
        O_ref, L_ref = orc.varlen_forward(*args, one_q, one_k, d["scale"], True)
        check_o(np64(o[q0:q1]), O_ref, f"O seq {b}")
        check_lse(np64(lse[:, q0:q1]), L_ref, f"LSE seq {b}")
        dQ, dK, dV = orc.varlen_backward(*args, np64(d["do"][q0:q1]), one_q, one_k, d["scale"], True)
        check_grad(np64(dq[q0:q1]), dQ, f"dQ seq {b}")
        check_grad(np64(dk[k0:k1]), dK, f"dK seq {b}")
        check_grad(np64(dv[k0:k1]), dV, f"dV seq {b}")
