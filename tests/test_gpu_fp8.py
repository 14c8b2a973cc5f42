"""GPU parity: the FP8 (e4m3) input forward against the fp64 oracle.

The oracle computes exact attention over the dequantized inputs. The kernel
rounds P to e4m3 before P V, so the bound is derived from that rounding: an
e4m3 value in the normal range (>= 2^-6) is within 2^-4 of x relatively, a
subnormal within 2^-10 absolutely; the kernel normalises by its fp32 row sum l
taken relative to a running maximum that never exceeds the true one, so
l >= l_true = sum_j exp(s_ij - max_i) and, per element,
  |O - O_ref|_id <= 2^-4 sum_j P_ij |V_jd| + 2^-10 sum_j |V_jd| / l_true_i
                    + 2^-8 |O_ref_id| (bf16 output) + 1e-3 (fp32 arithmetic).
The first sum is the oracle run on |V|. Independent roundings rarely add up
to that worst case, so the mean error must also stay below half the mean
bound. LSE does not involve the rounded P: max|diff| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs
from tests.parity import check_lse, fp8_error_bound, np64

pytestmark = pytest.mark.gpu


def _run(d, causal):
    q, k, v, off = (d[x].cuda() for x in ("q", "k", "v", "offsets"))
    o, lse = jfa.jfa_fwd_fp8(q, k, v, off, d["max_seqlen"], d["q_descale"], d["k_descale"], d["v_descale"],
                             d["scale"], causal, check=True)
    torch.cuda.synchronize()
    return np64(o), np64(lse)


def _check(d, causal, tag):
    o, lse = _run(d, causal)
    qd, kd, vd = d["q_descale"], d["k_descale"], d["v_descale"]
    q8, k8, v8 = (d[x].numpy() for x in ("q", "k", "v"))
    off = d["offsets"].numpy()
    O_ref, L_ref = orc.attention_forward_fp8(q8, k8, v8, off, d["scale"], causal, qd, kd, vd)
    check_lse(lse, L_ref, f"LSE {tag}")
    # the bound's terms, from the dequantized inputs
    q, k, v = orc.e4m3_decode(q8) * qd, orc.e4m3_decode(k8) * kd, orc.e4m3_decode(v8) * vd
    bound = fp8_error_bound(q, k, v, off, d["scale"], causal, O_ref)
    err = np.abs(o - O_ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"O {tag}: |diff| {err[worst]:.3e} > bound {bound[worst]:.3e}"
    assert err.mean() <= 0.5 * bound.mean(), f"O {tag}: mean |diff| {err.mean():.3e} vs mean bound {bound.mean():.3e}"


EDGE = [1, 127, 128, 129, 0, 255, 256, 300, 64, 513]


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_edge_lengths(causal):
    d = inputs.fp8_from_lengths(EDGE, 2, seed=61)
    _check(d, causal, f"edges causal={causal}")


def test_fp8_gem_like_reduced_batch():
    """GEM-like lengths (max_len 1024, sparsity 0.5, H = 4) on 24 sequences."""
    g = torch.Generator().manual_seed(62)
    lengths = inputs.uniform_lengths(24, 1, 1024, g)
    d = inputs.fp8_from_lengths(lengths, 4, seed=63)
    _check(d, False, "gem-like")


def test_fp8_descales_scale_the_output():
    """Doubling v_descale doubles O exactly (up to bf16 rounding of the same values);
    scaling k_descale by c equals scaling the softmax scale by c."""
    d = inputs.fp8_from_lengths([200, 77], 2, seed=64)
    q, k, v, off = (d[x].cuda() for x in ("q", "k", "v", "offsets"))
    o1, l1 = jfa.jfa_fwd_fp8(q, k, v, off, 200, 1.0, 1.0, 1.0, 0.05, check=True)
    o2, l2 = jfa.jfa_fwd_fp8(q, k, v, off, 200, 1.0, 1.0, 2.0, 0.05, check=True)
    o3, l3 = jfa.jfa_fwd_fp8(q, k, v, off, 200, 1.0, 2.0, 1.0, 0.025, check=True)
    assert torch.equal(o2, (2 * o1.float()).to(torch.bfloat16)) and torch.equal(l1, l2)
    assert torch.equal(o3, o1) and torch.equal(l3, l1)


def _vt_reference(v_bf16, offsets, heads, inv):
    """The V blocks jfa_fp8_quantize_v writes, built on the CPU: e4m3(v * inv) with torch's
    round-to-nearest conversion, block (tile_base[b] + t) * H + h holding [d][key] of key tile t."""
    codes = (v_bf16.float() * torch.tensor(inv, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    off = [int(x) for x in offsets]
    blocks = []
    for b in range(len(off) - 1):
        L = off[b + 1] - off[b]
        for t in range((L + 127) // 128):
            rows = min(128, L - 128 * t)
            for h in range(heads):
                blk = torch.zeros((128, 128), dtype=torch.uint8)
                blk[:, :rows] = codes[off[b] + 128 * t:off[b] + 128 * t + rows, h, :].T
                blocks.append(blk)
    return torch.stack(blocks).reshape(-1) if blocks else torch.zeros(0, dtype=torch.uint8)


def test_fp8_quantize_v_layout_bit_exact():
    """jfa_fp8_quantize_v: every byte of every block equals the CPU quantization placed by the
    documented layout (zeros past the end of a sequence)."""
    g = torch.Generator().manual_seed(64)
    lengths = torch.tensor(EDGE, dtype=torch.int32)
    d = inputs.jagged_from_lengths(lengths, 2, 128, g)
    v = d["v"]
    descale = float(v.float().abs().max()) / 440.0
    inv = float(np.float32(1.0) / np.float32(descale))
    vt = jfa.jfa_fp8_quantize_v(v.cuda(), d["offsets"].cuda(), d["max_seqlen"], descale, check=True)
    ref = _vt_reference(v, d["offsets"], 2, inv)
    got = vt.cpu()[:ref.numel()]
    assert torch.equal(got, ref), f"{int((got != ref).sum())} of {ref.numel()} bytes differ"


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_from_quantized_v_blocks(causal):
    """jfa_fwd_fp8 reading the blocks of jfa_fp8_quantize_v (no pass over V in the call) gives
    bit for bit the outputs of the call that takes the same e4m3 V and transposes it itself."""
    g = torch.Generator().manual_seed(65)
    lengths = inputs.uniform_lengths(24, 1, 1024, g)
    d = inputs.jagged_from_lengths(lengths, 4, 128, g)
    qd = kd = 0.02
    vd = float(d["v"].float().abs().max()) / 440.0
    q8 = (d["q"].float() / qd).clamp(-440, 440).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    k8 = (d["k"].float() / kd).clamp(-440, 440).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    inv = torch.tensor(float(np.float32(1.0) / np.float32(vd)), dtype=torch.float32)
    v8 = (d["v"].float() * inv).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    off = d["offsets"].cuda()
    o1, l1 = jfa.jfa_fwd_fp8(q8, k8, v8, off, d["max_seqlen"], qd, kd, vd, d["scale"], causal, check=True)
    vt = jfa.jfa_fp8_quantize_v(d["v"].cuda(), off, d["max_seqlen"], vd, check=True)
    o2, l2 = jfa.jfa_fwd_fp8(q8, k8, None, off, d["max_seqlen"], qd, kd, vd, d["scale"], causal, check=True, vt=vt)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
