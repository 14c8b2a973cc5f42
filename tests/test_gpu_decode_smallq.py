"""GPU parity: paged split-KV decode of a few query tokens per sequence.

The q_len new tokens of each sequence are its last q_len cache positions and
see the keys up to their own position. Compared with the fp64 oracle element
by element for GQA groups 1-16 with up to 16 (token, head) rows per KV head,
page sizes 1 / 16 / 128, fixed and per-sequence split counts, and sequences
shorter than q_len (rows that see no key); split bounds and counts bit for
bit; q_len 1 against the one-token entry point bit for bit; the full decode
workload with four query tokens on every sequence.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _run(d, splits, min_split=0):
    q, kc, vc = d["q"].cuda(), d["k_cache"].cuda(), d["v_cache"].cuda()
    pt, sl = d["page_table"].cuda(), d["seqlens_k"].cuda()
    B = d["batch"]
    bounds = torch.full((B, splits, 2), -1, dtype=torch.int32, device="cuda")
    counts = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    o, lse = jfa.jfa_decode_smallq(q, kc, vc, pt, sl, splits, min_split, d["scale"], split_bounds=bounds,
                                   split_counts=counts, check=True)
    torch.cuda.synchronize()
    return o, lse, bounds.cpu().numpy(), counts.cpu().numpy()


def _oracle(d, batch_ids=None):
    return orc.decode_smallq_forward(np64(d["q"]), np64(d["k_cache"]), np64(d["v_cache"]), d["page_table"].numpy(),
                                     d["seqlens_k"].numpy(), d["page_size"], d["scale"], batch_ids)


LENS = [0, 1, 2, 3, 15, 16, 17, 100, 1000, 333]


@pytest.mark.parametrize("kv_heads,q_len", [(8, 4), (4, 2), (16, 2), (32, 1), (2, 1), (8, 3), (16, 1)])
@pytest.mark.parametrize("page_size", [1, 16, 128])
def test_smallq_ragged(kv_heads, q_len, page_size):
    # 32 query heads: group 32 / kv_heads, rows of a tile = group x q_len (<= 16)
    d = inputs.decode_inputs(q_heads=32, kv_heads=kv_heads, page_size=page_size, seed=51, seqlens=LENS, q_len=q_len)
    O_ref, L_ref = _oracle(d)
    for splits, mn in ((1, 0), (3, 0), (16, 0), (16, 64)):
        o, lse, bounds, counts = _run(d, splits, mn)
        tag = f"Hkv={kv_heads} q_len={q_len} P={page_size} S={splits} min={mn}"
        check_o(np64(o), O_ref, f"O {tag}")
        check_lse(np64(lse), L_ref, f"LSE {tag}")
        exp_counts = orc.split_counts(d["seqlens_k"].numpy(), splits, mn)
        assert counts.tolist() == exp_counts.tolist(), tag
        assert (bounds == orc.split_bounds_per_seq(d["seqlens_k"].numpy(), splits, exp_counts)).all(), tag


def test_smallq_rows_without_keys():
    """Sequences shorter than q_len: the first q_len - L tokens see no key."""
    d = inputs.decode_inputs(q_heads=8, kv_heads=2, page_size=16, seed=52, seqlens=[1, 2, 0, 4], q_len=4)
    o, lse, _, _ = _run(d, 2)
    O_ref, L_ref = _oracle(d)
    check_o(np64(o), O_ref, "O short")
    check_lse(np64(lse), L_ref, "LSE short")
    assert np.isneginf(np64(lse)[0, :3]).all() and (np64(o)[0, :3] == 0).all()


def test_smallq_one_token_equals_decode():
    """q_len 1 runs the same split kernel as jfa_decode_splitkv: identical bits."""
    d = inputs.decode_inputs(batch=6, q_heads=32, kv_heads=8, lk_lo=10, lk_hi=3000, page_size=16, seed=53, q_len=1)
    o, lse, _, _ = _run(d, 8)
    q1 = d["q"][:, 0].contiguous().cuda()
    o1, lse1 = jfa.jfa_decode_splitkv(q1, d["k_cache"].cuda(), d["v_cache"].cuda(), d["page_table"].cuda(),
                                      d["seqlens_k"].cuda(), 8, d["scale"], check=True)
    assert torch.equal(o[:, 0], o1) and torch.equal(lse[:, 0], lse1)


@pytest.mark.parametrize("min_split", [0, 1024])
def test_smallq_full_size(min_split):
    """Decode workload (batch 32, Hq 32 / Hkv 8, L_k U[1024, 32768], page 16) with four
    query tokens; the oracle checks every row of every sequence."""
    d = inputs.decode_inputs(page_size=16, seed=0, q_len=4)
    o, lse, bounds, counts = _run(d, 16, min_split)
    O_ref, L_ref = _oracle(d)
    check_o(np64(o), O_ref, "O full")
    check_lse(np64(lse), L_ref, "LSE full")
    exp_counts = orc.split_counts(d["seqlens_k"].numpy(), 16, min_split)
    assert counts.tolist() == exp_counts.tolist()
    assert (bounds == orc.split_bounds_per_seq(d["seqlens_k"].numpy(), 16, exp_counts)).all()
