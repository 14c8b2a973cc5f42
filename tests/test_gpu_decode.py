"""GPU parity: split-KV paged GQA decode against the fp64 oracle.

Covers page sizes 1 / 3 / 16 / 128, split counts 1 .. 128, GQA groups 1 .. 16,
empty / length-1 / ragged sequences, the full-size decode workload (every
sequence), and bit-exact split bounds.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _run(d, splits, bounds=True, check=True):
    q, kc, vc = d["q"].cuda(), d["k_cache"].cuda(), d["v_cache"].cuda()
    pt, sl = d["page_table"].cuda(), d["seqlens_k"].cuda()
    B = q.shape[0]
    sb = torch.full((B, splits, 2), -7, dtype=torch.int32, device="cuda") if bounds else None
    o, lse = jfa.jfa_decode_splitkv(q, kc, vc, pt, sl, splits, d["scale"], split_bounds=sb, check=check)
    torch.cuda.synchronize()
    return o, lse, sb


def _oracle(d, batch_ids=None):
    return orc.decode_forward(np64(d["q"]), np64(d["k_cache"]), np64(d["v_cache"]), d["page_table"].numpy(),
                              d["seqlens_k"].numpy(), d["page_size"], d["scale"], batch_ids=batch_ids)


@pytest.mark.parametrize("page_size", [1, 3, 16, 128])
def test_decode_small_ragged(page_size):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2049]
    d = inputs.decode_inputs(q_heads=32, kv_heads=8, page_size=page_size, seed=3, seqlens=lens)
    O_ref, L_ref = _oracle(d)
    for S in (1, 2, 5, 16, 64, 128):
        o, lse, sb = _run(d, S)
        check_o(np64(o), O_ref, f"O (P={page_size}, S={S})")
        check_lse(np64(lse), L_ref, f"LSE (P={page_size}, S={S})")
        assert sb.cpu().numpy().tolist() == orc.split_bounds(np.array(lens), S).tolist()


@pytest.mark.parametrize("kv_heads", [16, 8, 4, 2, 1])
def test_decode_gqa_groups(kv_heads):
    lens = [37, 300, 1, 129]
    d = inputs.decode_inputs(q_heads=16, kv_heads=kv_heads, page_size=16, seed=4, seqlens=lens)
    O_ref, L_ref = _oracle(d)
    for S in (1, 3):
        o, lse, _ = _run(d, S)
        check_o(np64(o), O_ref, f"O (Hkv={kv_heads}, S={S})")
        check_lse(np64(lse), L_ref, f"LSE (Hkv={kv_heads}, S={S})")


@pytest.mark.parametrize("page_size", [1, 16, 128])
def test_decode_full_size(page_size):
    """Batch 32, 32 Q heads / 8 KV heads, KV lengths uniform in [1024, 32768]:
    every sequence against the oracle, at three split counts."""
    d = inputs.decode_inputs(page_size=page_size, seed=0)
    O_ref, L_ref = _oracle(d)
    lens = d["seqlens_k"].numpy()
    for S in (1, 16, 64):
        o, lse, sb = _run(d, S)
        check_o(np64(o), O_ref, f"O (P={page_size}, S={S})")
        check_lse(np64(lse), L_ref, f"LSE (P={page_size}, S={S})")
        assert sb.cpu().numpy().tolist() == orc.split_bounds(lens, S).tolist()


def test_decode_bad_page_table_is_reported():
    """A page index past num_pages is reported as JFA_ERR_BAD_INPUT (the kernel
    substitutes page 0 and keeps every access in bounds)."""
    d = inputs.decode_inputs(q_heads=8, kv_heads=2, page_size=4, seed=5, seqlens=[9, 4])
    d["page_table"][0, 1] = d["num_pages"] + 5
    with pytest.raises(jfa.JfaError) as ei:
        _run(d, 2, bounds=False, check=True)
    assert ei.value.status == 6
