"""The entry points inside a CUDA graph.

Every call enqueues only stream-ordered work (a status-clear kernel, the
queue build, the kernels, each later kernel launched as a programmatic
dependent of the one before) after host-side argument checks and tensor-map
encoding, so a step with fixed shapes, pointers and workspaces can be captured
once and replayed: small, launch-bound batches then cost one graph launch per
step. Each replay here reads fresh values copied into the captured input
tensors and is compared with the oracle.
"""
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_grad, check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _new_values(d, seed):
    g = torch.Generator().manual_seed(seed)
    return {k: torch.randn(d[k].shape, generator=g).to(torch.bfloat16) for k in ("q", "k", "v", "do")}


def test_fwd_bwd_replayed_from_a_cuda_graph():
    lengths = [70, 130, 5, 256]
    g0 = torch.Generator().manual_seed(71)
    d = inputs.jagged_from_lengths(torch.tensor(lengths, dtype=torch.int32), 2, 64, g0)
    dev = {k: d[k].cuda() for k in ("q", "k", "v", "do", "offsets")}
    o, lse = torch.empty_like(dev["q"]), torch.empty((2, d["total"]), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(dev["q"]) for _ in range(3))
    ws_f = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")

    def step():
        jfa.jfa_fwd(dev["q"], dev["k"], dev["v"], dev["offsets"], d["max_seqlen"], d["scale"], True, o=o, lse=lse,
                    workspace=ws_f)
        jfa.jfa_bwd(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, dev["offsets"], d["max_seqlen"], d["scale"],
                    True, dq=dq, dk=dk, dv=dv, workspace=ws_b)

    step()  # first calls set kernel attributes outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (72, 73):
        vals = _new_values(d, seed)
        for k, t in vals.items():
            dev[k].copy_(t)
        graph.replay()
        torch.cuda.synchronize()
        assert jfa.jfa_read_device_status(ws_b) == (0, 0)
        off = d["offsets"].numpy()
        args = [np64(vals[k]) for k in ("q", "k", "v")]
        O_ref, L_ref = orc.attention_forward(*args, off, d["scale"], True)
        check_o(np64(o), O_ref, f"graph O seed {seed}")
        check_lse(np64(lse), L_ref, f"graph LSE seed {seed}")
        dQ, dK, dV, _ = orc.attention_backward(*args, np64(vals["do"]), off, d["scale"], True)
        check_grad(np64(dq), dQ, f"graph dQ seed {seed}")
        check_grad(np64(dk), dK, f"graph dK seed {seed}")
        check_grad(np64(dv), dV, f"graph dV seed {seed}")


def test_decode_replayed_from_a_cuda_graph():
    """The decode chain (status clear, split kernel, merge kernel) in a graph."""
    d = inputs.decode_inputs(q_heads=8, kv_heads=2, page_size=16, seed=74, seqlens=[1, 100, 517, 2049])
    dev = {k: d[k].cuda() for k in ("q", "k_cache", "v_cache", "page_table", "seqlens_k")}
    o = torch.empty_like(dev["q"])
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")

    def step():
        jfa.jfa_decode_splitkv(dev["q"], dev["k_cache"], dev["v_cache"], dev["page_table"], dev["seqlens_k"], 4,
                               d["scale"], o=o, lse=lse, workspace=ws)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (75, 76):
        g = torch.Generator().manual_seed(seed)
        vals = {k: torch.randn(d[k].shape, generator=g).to(torch.bfloat16) for k in ("q", "k_cache", "v_cache")}
        for k, t in vals.items():
            dev[k].copy_(t)
        graph.replay()
        torch.cuda.synchronize()
        assert jfa.jfa_read_device_status(ws) == (0, 0)
        O_ref, L_ref = orc.decode_forward(np64(vals["q"]), np64(vals["k_cache"]), np64(vals["v_cache"]),
                                          d["page_table"].numpy(), d["seqlens_k"].numpy(), 16, d["scale"])
        check_o(np64(o), O_ref, f"graph decode O seed {seed}")
        check_lse(np64(lse), L_ref, f"graph decode LSE seed {seed}")


def test_broadcast_q_replayed_from_a_cuda_graph():
    """The broadcast-Q forward and backward chains in one graph; dQ is the sum over the batch."""
    d = inputs.broadcast_inputs(batch=3, q_len=40, heads=2, head_dim=64, lk_lo=1, lk_hi=300, seed=77)
    dev = {k: d[k].cuda() for k in ("q", "k", "v", "do", "kv_offsets")}
    mx = int(d["max_seqlen_k"])
    o, lse = jfa.jfa_fwd_broadcast_q(dev["q"], dev["k"], dev["v"], dev["kv_offsets"], mx, d["scale"])
    dq, dk, dv = torch.empty_like(dev["q"]), torch.empty_like(dev["k"]), torch.empty_like(dev["v"])
    ws_f = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")

    def step():
        jfa.jfa_fwd_broadcast_q(dev["q"], dev["k"], dev["v"], dev["kv_offsets"], mx, d["scale"], o=o, lse=lse,
                                workspace=ws_f)
        jfa.jfa_bwd_broadcast_q(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, dev["kv_offsets"], mx, d["scale"],
                                dq=dq, dk=dk, dv=dv, workspace=ws_b)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (78, 79):
        g = torch.Generator().manual_seed(seed)
        vals = {k: torch.randn(d[k].shape, generator=g).to(torch.bfloat16) for k in ("q", "k", "v", "do")}
        for k, t in vals.items():
            dev[k].copy_(t)
        graph.replay()
        torch.cuda.synchronize()
        assert jfa.jfa_read_device_status(ws_b) == (0, 0)
        off = d["kv_offsets"].numpy()
        args = [np64(vals[k]) for k in ("q", "k", "v")]
        O_ref, L_ref = orc.broadcast_forward(*args, off, d["scale"])
        check_o(np64(o), O_ref, f"graph broadcast O seed {seed}")
        check_lse(np64(lse), L_ref, f"graph broadcast LSE seed {seed}")
        dQ, dK, dV = orc.broadcast_backward(*args, np64(vals["do"]), off, d["scale"])
        check_grad(np64(dq), dQ, f"graph broadcast dQ seed {seed}")
        check_grad(np64(dk), dK, f"graph broadcast dK seed {seed}")
        check_grad(np64(dv), dV, f"graph broadcast dV seed {seed}")
