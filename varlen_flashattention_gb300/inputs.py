"""Seeded synthetic inputs for the jagged attention workloads.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path (through the binding) and the fp64
oracle consume the tensors it returns, so it is the one piece they share.

All draws use a CPU ``torch.Generator`` seeded explicitly, in a fixed order, so
the same seed gives the same bf16 tensors on every machine:

* jagged self-attention: lengths -> Q -> K -> V -> dO
* broadcast-Q:           lengths -> Q -> K -> V -> dO
* varlen / GQA:          query lengths -> key lengths -> Q -> K -> V -> dO
* paged decode:          kv lengths -> page permutation -> Q -> K cache -> V cache

Values are ``torch.randn`` in fp32, then rounded to bf16; the identical bf16
tensors go to the GPU and (upcast exactly to fp64) to the oracle.

Sequence lengths for the "sparsity" sweep of the jagged workloads (Meta's
jagged attention post, which sweeps sparsity 0.1 / 0.5 / 0.9 but gives no
formula): mean fill f = 1 - sparsity of ``max_len``, lengths uniform integers
in [lo, hi] with
  f >= 0.5: lo = round((2f - 1) * max_len), hi = max_len
  f <  0.5: lo = 1,                         hi = round(2f * max_len)
so sparsity 0.5 is exactly "uniform in [1, max_len]".
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def randn_bf16_device(shape, seed: int, device) -> torch.Tensor:
    """N(0,1) values rounded to bf16, drawn directly on `device` with its own
    seeded generator. Used where only the shape and distribution matter (the
    benchmark) and where a CPU draw would be too large (the test past 2^31
    elements, which copies its sampled sequences back for the oracle); other
    parity tests use the CPU draws above."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def sparsity_range(max_len: int, sparsity: float) -> tuple[int, int]:
    """Inclusive [lo, hi] of the uniform length draw for a sparsity level."""
    f = 1.0 - float(sparsity)
    if f >= 0.5:
        lo = int(round((2.0 * f - 1.0) * max_len))
        hi = int(max_len)
    else:
        lo = 1
        hi = int(round(2.0 * f * max_len))
    return max(lo, 1), max(hi, 1)


def uniform_lengths(batch: int, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """int32 [batch] uniform integers in [lo, hi]."""
    return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64).to(torch.int32)


def offsets_from_lengths(lengths: torch.Tensor) -> torch.Tensor:
    """int32 [B+1] exclusive prefix sum: offsets[0] = 0, offsets[B] = total."""
    off = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    assert int(off[-1]) < 2**31
    return off.to(torch.int32)


def jagged_from_lengths(lengths, heads: int, head_dim: int, g: torch.Generator,
                        with_grad: bool = True) -> dict:
    lengths = torch.as_tensor(lengths, dtype=torch.int32)
    offsets = offsets_from_lengths(lengths)
    total = int(offsets[-1])
    shape = (total, heads, head_dim)
    out = {
        "lengths": lengths,
        "offsets": offsets,
        "total": total,
        "max_seqlen": int(lengths.max()) if lengths.numel() else 0,
        "heads": heads,
        "head_dim": head_dim,
        "scale": 1.0 / math.sqrt(head_dim),
        "q": _randn_bf16(shape, g),
        "k": _randn_bf16(shape, g),
        "v": _randn_bf16(shape, g),
    }
    if with_grad:
        out["do"] = _randn_bf16(shape, g)
    return out


def jagged_inputs(batch: int, max_len: int, sparsity: float, heads: int, head_dim: int,
                  seed: int = 0, with_grad: bool = True) -> dict:
    """GEM-like jagged self-attention: lengths by the sparsity reading above."""
    g = _gen(seed)
    lo, hi = sparsity_range(max_len, sparsity)
    lengths = uniform_lengths(batch, lo, hi, g)
    out = jagged_from_lengths(lengths, heads, head_dim, g, with_grad)
    out["causal"] = False
    return out


def tiny_inputs(seed: int = 0) -> dict:
    """Tiny jagged case: batch 4, lengths uniform in [1, 64], 2 heads, head_dim 64."""
    g = _gen(seed)
    lengths = uniform_lengths(4, 1, 64, g)
    out = jagged_from_lengths(lengths, 2, 64, g, True)
    out["causal"] = False
    return out


def dense_causal_inputs(batch: int = 4, seqlen: int = 8192, heads: int = 16, head_dim: int = 128,
                        seed: int = 0) -> dict:
    """Dense LLM-style causal case, packed as equal-length jagged sequences."""
    g = _gen(seed)
    lengths = torch.full((batch,), seqlen, dtype=torch.int32)
    out = jagged_from_lengths(lengths, heads, head_dim, g, True)
    out["causal"] = True
    return out


def varlen_from_lengths(q_lengths, k_lengths, q_heads: int, kv_heads: int, head_dim: int,
                        g: torch.Generator, with_grad: bool = True) -> dict:
    """Varlen / GQA case from given lengths: Q, dO [total_q, Hq, d]; K, V [total_k, Hkv, d]."""
    q_lengths = torch.as_tensor(q_lengths, dtype=torch.int32)
    k_lengths = torch.as_tensor(k_lengths, dtype=torch.int32)
    assert q_lengths.numel() == k_lengths.numel()
    qo, ko = offsets_from_lengths(q_lengths), offsets_from_lengths(k_lengths)
    tq, tk = int(qo[-1]), int(ko[-1])
    out = {
        "q_lengths": q_lengths, "k_lengths": k_lengths,
        "q_offsets": qo, "k_offsets": ko,
        "total_q": tq, "total_k": tk,
        "max_seqlen_q": int(q_lengths.max()) if q_lengths.numel() else 0,
        "max_seqlen_k": int(k_lengths.max()) if k_lengths.numel() else 0,
        "q_heads": q_heads, "kv_heads": kv_heads, "head_dim": head_dim,
        "scale": 1.0 / math.sqrt(head_dim),
        "q": _randn_bf16((tq, q_heads, head_dim), g),
        "k": _randn_bf16((tk, kv_heads, head_dim), g),
        "v": _randn_bf16((tk, kv_heads, head_dim), g),
    }
    if with_grad:
        out["do"] = _randn_bf16((tq, q_heads, head_dim), g)
    return out


def varlen_inputs(batch: int, q_lo: int, q_hi: int, k_lo: int, k_hi: int, q_heads: int, kv_heads: int,
                  head_dim: int, seed: int = 0, with_grad: bool = True) -> dict:
    """Varlen / GQA case: query lengths U[q_lo, q_hi], key lengths U[k_lo, k_hi] drawn independently."""
    g = _gen(seed)
    ql = uniform_lengths(batch, q_lo, q_hi, g)
    kl = uniform_lengths(batch, k_lo, k_hi, g)
    return varlen_from_lengths(ql, kl, q_heads, kv_heads, head_dim, g, with_grad)


def fp8_quantize(x: torch.Tensor):
    """Per-tensor e4m3 quantization of fp32 values: descale = amax / 448 (the largest e4m3
    value), codes = e4m3(x / descale) as uint8. Returns (codes, descale)."""
    amax = float(x.abs().max()) if x.numel() else 1.0
    descale = max(amax, 1e-30) / 448.0
    codes = (x / descale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, descale


def fp8_from_lengths(lengths, heads: int, seed: int, head_dim: int = 128) -> dict:
    """FP8 jagged inputs: lengths -> Q -> K -> V drawn N(0,1) in fp32, each quantized to e4m3
    with its own descale."""
    g = _gen(seed)
    lengths = torch.as_tensor(lengths, dtype=torch.int32)
    offsets = offsets_from_lengths(lengths)
    total = int(offsets[-1])
    out = {"lengths": lengths, "offsets": offsets, "total": total,
           "max_seqlen": int(lengths.max()) if lengths.numel() else 0, "heads": heads, "head_dim": head_dim,
           "scale": 1.0 / math.sqrt(head_dim)}
    for name in ("q", "k", "v"):
        x = torch.randn(total, heads, head_dim, generator=g, dtype=torch.float32)
        out[name], out[name + "_descale"] = fp8_quantize(x)
    return out


def broadcast_inputs(batch: int = 512, q_len: int = 256, heads: int = 4, head_dim: int = 128,
                     lk_lo: int = 16, lk_hi: int = 2048, seed: int = 0) -> dict:
    """Broadcast-Q: one dense Q [q_len, H, d] shared by `batch` jagged K/V sequences."""
    g = _gen(seed)
    lengths = uniform_lengths(batch, lk_lo, lk_hi, g)
    offsets = offsets_from_lengths(lengths)
    total = int(offsets[-1])
    return {
        "lengths": lengths,
        "kv_offsets": offsets,
        "total_k": total,
        "max_seqlen_k": int(lengths.max()) if batch else 0,
        "batch": batch,
        "q_len": q_len,
        "heads": heads,
        "head_dim": head_dim,
        "scale": 1.0 / math.sqrt(head_dim),
        "q": _randn_bf16((q_len, heads, head_dim), g),
        "k": _randn_bf16((total, heads, head_dim), g),
        "v": _randn_bf16((total, heads, head_dim), g),
        "do": _randn_bf16((batch, q_len, heads, head_dim), g),
    }


def decode_inputs(batch: int = 32, q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128,
                  lk_lo: int = 1024, lk_hi: int = 32768, page_size: int = 16, seed: int = 0,
                  seqlens=None, q_len=None) -> dict:
    """Paged GQA decode: one query token per sequence, KV cache in pages of
    `page_size` tokens, pages handed out by a random permutation.

    Layouts: q [B, Hq, d]; k_cache / v_cache [num_pages, page_size, Hkv, d];
    page_table int32 [B, max_pages] (entries past ceil(L_b / page_size) are 0
    and never read); seqlens_k int32 [B].
    """
    g = _gen(seed)
    if seqlens is None:
        seqlens = uniform_lengths(batch, lk_lo, lk_hi, g)
    else:
        seqlens = torch.as_tensor(seqlens, dtype=torch.int32)
        batch = seqlens.numel()
    pages_per_seq = [(int(l) + page_size - 1) // page_size for l in seqlens.tolist()]
    num_pages = max(sum(pages_per_seq), 1)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    max_pages = max(max(pages_per_seq) if pages_per_seq else 1, 1)
    page_table = torch.zeros((batch, max_pages), dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        page_table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    # one query token per sequence ([B, Hq, d]), or q_len new tokens ([B, q_len, Hq, d])
    q = _randn_bf16((batch, q_heads, head_dim) if q_len is None else (batch, q_len, q_heads, head_dim), g)
    k_cache = _randn_bf16((num_pages, page_size, kv_heads, head_dim), g)
    v_cache = _randn_bf16((num_pages, page_size, kv_heads, head_dim), g)
    return {
        "batch": batch,
        "q_heads": q_heads,
        "kv_heads": kv_heads,
        "head_dim": head_dim,
        "page_size": page_size,
        "num_pages": num_pages,
        "max_pages": max_pages,
        "scale": 1.0 / math.sqrt(head_dim),
        "seqlens_k": seqlens,
        "page_table": page_table,
        "q": q,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "q_len": 1 if q_len is None else q_len,
    }
