"""Host-side argument checks of the Python binding (no GPU needed).

The kernels address every buffer from the shapes of q (and k), so the
binding rejects any tensor whose dtype, shape or layout disagrees with them,
and any tensor on another device, before anything reaches the library. These
tests pass CPU tensors: shape errors must be raised first, and a call whose
shapes are all right must still refuse to run off the GPU.
"""
import pytest
import torch

import varlen_flashattention_gb300 as jfa

bf16, f32, i32 = torch.bfloat16, torch.float32, torch.int32


def _self(total=10, H=2, d=64):
    q = torch.zeros(total, H, d, dtype=bf16)
    return dict(q=q, k=q.clone(), v=q.clone(), o=q.clone(), dout=q.clone(), lse=torch.zeros(H, total, dtype=f32),
                offsets=torch.tensor([0, 4, total], dtype=i32))


def _bwd(t, **over):
    a = dict(t, **over)
    return jfa.jfa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["offsets"], 8,
                       dq=a.get("dq"), dk=a.get("dk"), dv=a.get("dv"))


def test_bwd_rejects_mismatched_shapes():
    t = _self()
    with pytest.raises(ValueError, match="k must have shape"):
        _bwd(t, k=torch.zeros(9, 2, 64, dtype=bf16))
    with pytest.raises(ValueError, match="lse must have shape"):
        _bwd(t, lse=torch.zeros(2, 9, dtype=f32))
    with pytest.raises(ValueError, match="dout must have shape"):
        _bwd(t, dout=torch.zeros(10, 2, 128, dtype=bf16))
    with pytest.raises(TypeError, match="o must be torch.bfloat16"):
        _bwd(t, o=torch.zeros(10, 2, 64, dtype=f32))
    with pytest.raises(ValueError, match="offsets must hold"):
        _bwd(t, offsets=torch.zeros(0, dtype=i32))
    with pytest.raises(ValueError, match="v must be contiguous"):
        _bwd(t, v=torch.zeros(10, 64, 2, dtype=bf16).transpose(1, 2))


def test_bwd_rejects_host_tensors():
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        _bwd(_self())


def test_fwd_rejects_mismatched_outputs():
    t = _self()
    with pytest.raises(ValueError, match="v must have shape"):
        jfa.jfa_fwd(t["q"], t["k"], torch.zeros(10, 2, 32, dtype=bf16), t["offsets"], 8)
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        jfa.jfa_fwd(t["q"], t["k"], t["v"], t["offsets"], 8, o=torch.zeros(10, 2, 64, dtype=bf16))


def test_varlen_rejects_mismatched_shapes():
    q = torch.zeros(12, 4, 64, dtype=bf16)
    k = torch.zeros(20, 2, 64, dtype=bf16)
    qo = torch.tensor([0, 5, 12], dtype=i32)
    ko = torch.tensor([0, 9, 20], dtype=i32)
    with pytest.raises(ValueError, match="v must have shape"):
        jfa.jfa_fwd_varlen(q, k, torch.zeros(20, 4, 64, dtype=bf16), qo, ko, 7, 11)
    with pytest.raises(ValueError, match="k must have shape"):
        jfa.jfa_fwd_varlen(q, torch.zeros(20, 2, 128, dtype=bf16), k, qo, ko, 7, 11)
    with pytest.raises(ValueError, match="same length"):
        jfa.jfa_fwd_varlen(q, k, k, qo, torch.tensor([0, 20], dtype=i32), 7, 11)
    lse = torch.zeros(4, 12, dtype=f32)
    with pytest.raises(ValueError, match="lse must have shape"):
        jfa.jfa_bwd_varlen(q, k, k, q, q, lse[:2], qo, ko, 7, 11)
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        jfa.jfa_bwd_varlen(q, k, k, q, q, lse, qo, ko, 7, 11)


def test_broadcast_rejects_mismatched_shapes():
    q = torch.zeros(256, 4, 128, dtype=bf16)
    k = torch.zeros(50, 4, 128, dtype=bf16)
    off = torch.tensor([0, 20, 50], dtype=i32)
    o = torch.zeros(2, 256, 4, 128, dtype=bf16)
    lse = torch.zeros(2, 4, 256, dtype=f32)
    with pytest.raises(ValueError, match="k must have shape"):
        jfa.jfa_fwd_broadcast_q(q, torch.zeros(50, 2, 128, dtype=bf16), k, off, 30)
    with pytest.raises(ValueError, match="o must have shape"):
        jfa.jfa_bwd_broadcast_q(q, k, k, o[:1], o, lse, off, 30)
    with pytest.raises(ValueError, match="lse must have shape"):
        jfa.jfa_bwd_broadcast_q(q, k, k, o, o, lse[:, :2], off, 30)
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        jfa.jfa_bwd_broadcast_q(q, k, k, o, o, lse, off, 30)


def test_decode_rejects_mismatched_shapes():
    q = torch.zeros(3, 8, 128, dtype=bf16)
    kc = torch.zeros(10, 16, 2, 128, dtype=bf16)
    pt = torch.zeros(3, 4, dtype=i32)
    sl = torch.ones(3, dtype=i32)
    with pytest.raises(ValueError, match="v_cache must have shape"):
        jfa.jfa_decode_splitkv(q, kc, kc[:5], pt, sl, 4)
    with pytest.raises(ValueError, match="page_table must have shape"):
        jfa.jfa_decode_splitkv(q, kc, kc, pt[:2], sl, 4)
    with pytest.raises(ValueError, match="seqlens_k must have shape"):
        jfa.jfa_decode_splitkv(q, kc, kc, pt, sl[:2], 4)
    with pytest.raises(ValueError, match="split_bounds must have shape"):
        jfa.jfa_decode_splitkv(q, kc, kc, pt, sl, 4, split_bounds=torch.zeros(3, 2, 2, dtype=i32))
    q4 = torch.zeros(3, 2, 8, 128, dtype=bf16)
    with pytest.raises(ValueError, match="split_counts must have shape"):
        jfa.jfa_decode_smallq(q4, kc, kc, pt, sl, 4, split_counts=torch.zeros(2, dtype=i32))
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        jfa.jfa_decode_smallq(q4, kc, kc, pt, sl, 4)


def test_fp8_rejects_mismatched_shapes():
    q = torch.zeros(10, 2, 128, dtype=torch.uint8)
    off = torch.tensor([0, 10], dtype=i32)
    with pytest.raises(ValueError, match="k must have shape"):
        jfa.jfa_fwd_fp8(q, q[:5], q, off, 10, 1.0, 1.0, 1.0)
    with pytest.raises(ValueError, match="lse must have shape"):
        jfa.jfa_fwd_fp8(q, q, q, off, 10, 1.0, 1.0, 1.0, lse=torch.zeros(2, 9, dtype=f32))


def test_bwd_rejects_mismatched_gradient_buffers():
    t = _self()
    with pytest.raises(ValueError, match="dk must have shape"):
        _bwd(t, dk=torch.zeros(10, 2, 32, dtype=bf16))
    with pytest.raises(TypeError, match="dq must be torch.bfloat16"):
        _bwd(t, dq=torch.zeros(10, 2, 64, dtype=f32))


def test_well_formed_host_buffers_reach_the_device_check():
    """Every entry point with correct shapes, outputs and gradient buffers
    passed in (on the host): the only complaint is the device."""
    t = _self()
    z = {n: torch.zeros_like(t["q"]) for n in ("dq", "dk", "dv")}
    calls = [
        lambda: jfa.jfa_fwd(t["q"], t["k"], t["v"], t["offsets"], 8, o=t["o"], lse=t["lse"]),
        lambda: _bwd(t, **z),
    ]
    q = torch.zeros(256, 4, 128, dtype=bf16)
    k = torch.zeros(50, 4, 128, dtype=bf16)
    off = torch.tensor([0, 20, 50], dtype=i32)
    o = torch.zeros(2, 256, 4, 128, dtype=bf16)
    lse = torch.zeros(2, 4, 256, dtype=f32)
    calls += [
        lambda: jfa.jfa_fwd_broadcast_q(q, k, k, off, 30, o=o, lse=lse),
        lambda: jfa.jfa_bwd_broadcast_q(q, k, k, o, o, lse, off, 30, dq=torch.zeros_like(q), dk=torch.zeros_like(k),
                                        dv=torch.zeros_like(k)),
    ]
    qv = torch.zeros(12, 4, 64, dtype=bf16)
    kv = torch.zeros(20, 2, 64, dtype=bf16)
    qo = torch.tensor([0, 5, 12], dtype=i32)
    ko = torch.tensor([0, 9, 20], dtype=i32)
    lv = torch.zeros(4, 12, dtype=f32)
    calls += [
        lambda: jfa.jfa_fwd_varlen(qv, kv, kv, qo, ko, 7, 11, o=torch.zeros_like(qv), lse=lv),
        lambda: jfa.jfa_bwd_varlen(qv, kv, kv, qv, qv, lv, qo, ko, 7, 11, dq=torch.zeros_like(qv),
                                   dk=torch.zeros_like(kv), dv=torch.zeros_like(kv)),
    ]
    q8 = torch.zeros(10, 2, 128, dtype=torch.uint8)
    calls.append(lambda: jfa.jfa_fwd_fp8(q8, q8, q8, torch.tensor([0, 10], dtype=i32), 10, 1.0, 1.0, 1.0,
                                         o=torch.zeros(10, 2, 128, dtype=bf16), lse=torch.zeros(2, 10, dtype=f32)))
    qd = torch.zeros(3, 8, 128, dtype=bf16)
    kc = torch.zeros(10, 16, 2, 128, dtype=bf16)
    pt = torch.zeros(3, 4, dtype=i32)
    sl = torch.ones(3, dtype=i32)
    q4 = torch.zeros(3, 2, 8, 128, dtype=bf16)
    calls += [
        lambda: jfa.jfa_decode_splitkv(qd, kc, kc, pt, sl, 4, o=torch.zeros_like(qd), lse=torch.zeros(3, 8),
                                       split_bounds=torch.zeros(3, 4, 2, dtype=i32)),
        lambda: jfa.jfa_decode_smallq(q4, kc, kc, pt, sl, 4, o=torch.zeros_like(q4), lse=torch.zeros(3, 2, 8),
                                      split_bounds=torch.zeros(3, 4, 2, dtype=i32),
                                      split_counts=torch.zeros(3, dtype=i32)),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="must be on a CUDA device"):
            call()


def test_fp8_vt_and_quantize_v_reject_mismatched_shapes():
    u8 = torch.uint8
    q = torch.zeros(10, 2, 128, dtype=u8)
    off = torch.tensor([0, 4, 10], dtype=i32)
    with pytest.raises(ValueError, match="vt must have shape"):  # the blocks of 2 sequences x 2 heads
        jfa.jfa_fwd_fp8(q, q, None, off, 8, 1.0, 1.0, 1.0, vt=torch.zeros(100, dtype=u8))
    with pytest.raises(TypeError, match="v must be torch.bfloat16"):
        jfa.jfa_fp8_quantize_v(q, off, 8, 1.0)
    v = torch.zeros(10, 2, 128, dtype=bf16)
    with pytest.raises(ValueError, match="vt must have shape"):
        jfa.jfa_fp8_quantize_v(v, off, 8, 1.0, vt=torch.zeros(7, dtype=u8))
    with pytest.raises(ValueError, match="must be on a CUDA device"):
        jfa.jfa_fp8_quantize_v(v, off, 8, 1.0)
