"""The seeded synthetic inputs (no GPU): the sparsity reading of the length
draws, determinism per seed, offsets, and the paged cache layout (every page
handed out exactly once)."""
import torch

from varlen_flashattention_gb300 import inputs


def test_sparsity_reading():
    # mean fill 1 - s of max_len, uniform lengths
    assert inputs.sparsity_range(1024, 0.1) == (819, 1024)
    assert inputs.sparsity_range(1024, 0.5) == (1, 1024)
    assert inputs.sparsity_range(1024, 0.9) == (1, 205)


def test_jagged_inputs_are_seeded_and_consistent():
    a = inputs.jagged_inputs(16, 1024, 0.9, 2, 64, seed=3)
    b = inputs.jagged_inputs(16, 1024, 0.9, 2, 64, seed=3)
    c = inputs.jagged_inputs(16, 1024, 0.9, 2, 64, seed=4)
    for key in ("lengths", "offsets", "q", "k", "v", "do"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["q"], c["q"])
    L, off = a["lengths"], a["offsets"]
    assert int(off[0]) == 0 and int(off[-1]) == a["total"] == int(L.sum())
    assert torch.equal(off[1:] - off[:-1], L)
    assert int(L.min()) >= 1 and int(L.max()) <= 205 and a["max_seqlen"] == int(L.max())
    assert a["q"].shape == (a["total"], 2, 64) and a["q"].dtype == torch.bfloat16


def test_paged_cache_hands_out_every_page_once():
    d = inputs.decode_inputs(batch=5, q_heads=8, kv_heads=2, page_size=16, seed=2, seqlens=[1, 0, 33, 16, 100])
    P = d["page_size"]
    used = []
    for b, L in enumerate(d["seqlens_k"].tolist()):
        n = (L + P - 1) // P
        used += d["page_table"][b, :n].tolist()
        assert d["page_table"][b, n:].eq(0).all()
    assert sorted(used) == list(range(d["num_pages"]))
    assert d["k_cache"].shape == (d["num_pages"], P, 2, 128)
