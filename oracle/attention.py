"""fp64 CPU oracle for jagged attention -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this module. The CUDA library never calls it, and it
imports nothing from the CUDA package: the two implementations share no code.

What it computes is exact attention and its exact gradient, written out from
the definitions, materialising S and P per (sequence, head) in fp64:

* Forward. "Cutting-edge isn't plug-and-play: customizing FA4 on B300"
  (TwelveLabs), section "FlashAttention recap": the score matrix is S = Q K^T
  and FlashAttention only tiles it, so the tiled result is mathematically
  equal to the naive one. Here: S = scale * Q K^T, P = softmax_rows(S),
  O = P V, and the saved log-sum-exp LSE_i = ln sum_j exp(S_ij) (natural log;
  the page only names "LSE").
* Jagged packing. "Optimizing Jagged Flash Attention with TLX" (aivexanews),
  third paragraph: sequences are packed back to back, boundaries kept in an
  offsets tensor, no padded tokens. Sequence b is rows offsets[b]:offsets[b+1].
* Backward. Same TwelveLabs page, section "Phase 2: chunked backward" and its
  pseudocode: S and dP are rebuilt per tile, P from S and the saved LSE, then
  dS from P, dP and "delta". As a plain gradient of O = softmax(scale Q K^T) V:
      dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id  ("delta"),
      dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
* Broadcast-Q. aivexanews page, third paragraph: one dense Q is shared by the
  whole batch, so dQ is the sum over the batch of the per-sequence dQ.
* Jagged attention with separate query and key lengths and grouped-query
  heads. "Cutting-edge isn't plug-and-play: customizing FA4 on B300"
  (TwelveLabs), section on why the development succeeded, second factor: the
  test suite the kernel had to pass spans MHA / GQA / MQA head layouts,
  causal and non-causal masks and varlen packing; "Optimizing FlashAttention-4
  for Efficient Inference" (hpjadul), section "PR 2186": several query heads
  share one KV head. Sequence b has its query rows at q_offsets[b] .. and its
  key rows at k_offsets[b] ..; query head h reads KV head h // (Hq / Hkv); dK
  and dV of a KV head sum over the query heads of its group.
* Paged split-KV GQA decode. "Optimizing FlashAttention-4 for Efficient
  Inference" (hpjadul), sections "PR 1940" (parallelism across the KV
  dimension), "PR 1999 and PR 2104" (arbitrary KV page sizes) and "PR 2186"
  (GQA packing). Attention of one query token per sequence against a KV cache
  addressed through a page table; query head h reads KV head h // (Hq / Hkv).
  The split/merge form is a second, separate function; its merge rule
  (lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s) is the plainest
  exact way to combine partial softmaxes and is not printed on the page.

Conventions where the pages are silent (readings, not statements of the pages):
  * an empty key set gives O = 0 and LSE = -inf (and zero gradients);
  * causal means L_q == L_k and key j is visible to query i iff j <= i;
  * with L_q != L_k (varlen functions), causal aligns the mask to the bottom
    right: key j is visible to query i iff j <= i + (L_k - L_q), so the last
    query sees every key; query rows that see no key get O = 0, LSE = -inf;
  * split bounds: c_b = ceil(L_b / S); split s covers [s c_b, min((s+1) c_b, L_b)).

Inputs are numpy arrays of float64 (bf16 values upcast exactly by the caller)
and integer offsets. Nothing here is blocked, fused or reordered beyond the
definitions above; numpy's matmul is the only library primitive used.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "seq_ranges", "attention_forward", "attention_backward",
    "broadcast_forward", "broadcast_backward",
    "split_bounds", "gather_paged", "decode_forward", "decode_split_partials",
    "merge_partials", "tile_queue",
    "lower_right_visible", "varlen_forward", "varlen_backward", "varlen_tile_queue",
    "split_counts", "split_bounds_per_seq", "decode_smallq_forward", "decode_smallq_split_partials",
    "e4m3_decode", "attention_forward_fp8",
]


def seq_ranges(offsets):
    """(start, end) of every packed sequence: rows offsets[b] .. offsets[b+1]."""
    off = [int(x) for x in np.asarray(offsets).reshape(-1)]
    return [(off[b], off[b + 1]) for b in range(len(off) - 1)]


def _softmax_rows(S):
    """Row softmax by definition, with the usual max shift for range.

    Returns (P, lse) with lse_i = ln sum_j exp(S_ij); rows whose scores are all
    -inf (no visible key) give P = 0 and lse = -inf."""
    m = np.max(S, axis=1, keepdims=True) if S.shape[1] else np.full((S.shape[0], 1), -np.inf)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    E = np.exp(S - m_safe)
    E[~np.broadcast_to(finite, E.shape)] = 0.0
    Z = np.sum(E, axis=1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(Z > 0, E / np.where(Z > 0, Z, 1.0), 0.0)
        lse = np.where(Z[:, 0] > 0, m_safe[:, 0] + np.log(np.where(Z[:, 0] > 0, Z[:, 0], 1.0)), -np.inf)
    return P, lse


def _scores(Qh, Kh, scale, causal):
    S = scale * (Qh @ Kh.T)
    if causal:
        Lq, Lk = S.shape
        assert Lq == Lk, "causal attention here is self-attention (L_q == L_k)"
        S = np.where(np.tril(np.ones((Lq, Lk), dtype=bool)), S, -np.inf)
    return S


def _head_forward(Qh, Kh, Vh, scale, causal):
    S = _scores(Qh, Kh, scale, causal)
    P, lse = _softmax_rows(S)
    return P @ Vh, lse, P


def _head_backward(Qh, Kh, Vh, dOh, scale, causal):
    """Exact gradient of O = softmax(scale Q K^T) V for one (sequence, head)."""
    S = _scores(Qh, Kh, scale, causal)
    P, _ = _softmax_rows(S)
    O = P @ Vh
    dV = P.T @ dOh
    dP = dOh @ Vh.T
    D = np.sum(dOh * O, axis=1)            # "delta": rowsum(dO * O)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ Kh)
    dK = scale * (dS.T @ Qh)
    return dQ, dK, dV, D


def attention_forward(q, k, v, offsets, scale, causal=False):
    """Jagged self-attention forward.

    q, k, v: [total, H, d] float64, packed by `offsets` (int [B+1]).
    Returns O [total, H, d] and LSE [H, total] (natural log)."""
    total, H, d = q.shape
    O = np.zeros((total, H, v.shape[2]), dtype=np.float64)
    LSE = np.full((H, total), -np.inf, dtype=np.float64)
    for s, e in seq_ranges(offsets):
        if e == s:
            continue
        for h in range(H):
            Oh, lse, _ = _head_forward(q[s:e, h], k[s:e, h], v[s:e, h], scale, causal)
            O[s:e, h] = Oh
            LSE[h, s:e] = lse
    return O, LSE


def attention_backward(q, k, v, do, offsets, scale, causal=False):
    """Jagged self-attention backward. Returns dQ, dK, dV [total, H, d] and
    D [H, total] (the "delta" row sums)."""
    total, H, d = q.shape
    dQ = np.zeros_like(q, dtype=np.float64)
    dK = np.zeros_like(k, dtype=np.float64)
    dV = np.zeros_like(v, dtype=np.float64)
    D = np.zeros((H, total), dtype=np.float64)
    for s, e in seq_ranges(offsets):
        if e == s:
            continue
        for h in range(H):
            a, b_, c, dd = _head_backward(q[s:e, h], k[s:e, h], v[s:e, h], do[s:e, h], scale, causal)
            dQ[s:e, h], dK[s:e, h], dV[s:e, h], D[h, s:e] = a, b_, c, dd
    return dQ, dK, dV, D


def broadcast_forward(q, k, v, kv_offsets, scale):
    """Broadcast-Q forward: q [Lq, H, d] is the query of every sequence b,
    k, v jagged [total_k, H, d]. Returns O [B, Lq, H, d], LSE [B, H, Lq]."""
    Lq, H, d = q.shape
    ranges = seq_ranges(kv_offsets)
    B = len(ranges)
    O = np.zeros((B, Lq, H, v.shape[2]), dtype=np.float64)
    LSE = np.full((B, H, Lq), -np.inf, dtype=np.float64)
    for b, (s, e) in enumerate(ranges):
        if e == s:
            continue
        for h in range(H):
            Oh, lse, _ = _head_forward(q[:, h], k[s:e, h], v[s:e, h], scale, False)
            O[b, :, h] = Oh
            LSE[b, h] = lse
    return O, LSE


def broadcast_backward(q, k, v, do, kv_offsets, scale):
    """Broadcast-Q backward: dQ [Lq, H, d] summed over the batch, dK and dV
    jagged [total_k, H, d]. do is [B, Lq, H, d]."""
    Lq, H, d = q.shape
    dQ = np.zeros_like(q, dtype=np.float64)
    dK = np.zeros_like(k, dtype=np.float64)
    dV = np.zeros_like(v, dtype=np.float64)
    for b, (s, e) in enumerate(seq_ranges(kv_offsets)):
        if e == s:
            continue
        for h in range(H):
            a, b_, c, _ = _head_backward(q[:, h], k[s:e, h], v[s:e, h], do[b, :, h], scale, False)
            dQ[:, h] += a
            dK[s:e, h] = b_
            dV[s:e, h] = c
    return dQ, dK, dV


# ----------------------------------------------------------------------------
# Paged split-KV GQA decode
# ----------------------------------------------------------------------------

def split_bounds(seqlens, num_splits):
    """int64 [B, S, 2]: (start, end) token range of every KV split.

    c_b = ceil(L_b / S); split s covers [s c_b, min((s+1) c_b, L_b)); a split
    whose start is at or past L_b is empty and reported as (L_b, L_b)."""
    seqlens = [int(x) for x in np.asarray(seqlens).reshape(-1)]
    S = int(num_splits)
    out = np.zeros((len(seqlens), S, 2), dtype=np.int64)
    for b, L in enumerate(seqlens):
        c = -(-L // S) if L > 0 else 0
        for s in range(S):
            lo = min(s * c, L)
            hi = min((s + 1) * c, L)
            out[b, s] = (lo, hi)
    return out


def gather_paged(cache, page_table_row, length, page_size):
    """Rows 0..length-1 of one sequence from a paged cache [num_pages, P, Hkv, d]:
    token t lives in page page_table_row[t // P], slot t % P."""
    idx_page = np.asarray([int(page_table_row[t // page_size]) for t in range(length)], dtype=np.int64)
    idx_slot = np.arange(length, dtype=np.int64) % page_size
    return cache[idx_page, idx_slot]           # [length, Hkv, d]


def _decode_one(qb, Kb, Vb, scale, q_heads, kv_heads):
    """One sequence: qb [Hq, d], Kb/Vb [L, Hkv, d] -> O [Hq, d], LSE [Hq]."""
    group = q_heads // kv_heads
    O = np.zeros((q_heads, Vb.shape[2] if Vb.ndim == 3 else qb.shape[1]), dtype=np.float64)
    LSE = np.full(q_heads, -np.inf, dtype=np.float64)
    if Kb.shape[0] == 0:
        return O, LSE
    for h in range(q_heads):
        g = h // group
        Oh, lse, _ = _head_forward(qb[h:h + 1], Kb[:, g], Vb[:, g], scale, False)
        O[h] = Oh[0]
        LSE[h] = lse[0]
    return O, LSE


def decode_forward(q, k_cache, v_cache, page_table, seqlens, page_size, scale, batch_ids=None):
    """Unsplit paged decode. q [B, Hq, d]; caches [num_pages, P, Hkv, d];
    returns O [B, Hq, d], LSE [B, Hq] (rows of `batch_ids` only, if given)."""
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    ids = range(B) if batch_ids is None else batch_ids
    O = np.zeros((B, Hq, d), dtype=np.float64)
    LSE = np.full((B, Hq), -np.inf, dtype=np.float64)
    for b in ids:
        L = int(seqlens[b])
        Kb = gather_paged(k_cache, page_table[b], L, page_size)
        Vb = gather_paged(v_cache, page_table[b], L, page_size)
        O[b], LSE[b] = _decode_one(q[b], Kb, Vb, scale, Hq, Hkv)
    return O, LSE


def decode_split_partials(q, k_cache, v_cache, page_table, seqlens, page_size, scale, num_splits):
    """Per-split partial results: O_s [S, B, Hq, d] (normalised within the
    split) and lse_s [S, B, Hq] (-inf for an empty split)."""
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    bounds = split_bounds(seqlens, num_splits)
    Os = np.zeros((num_splits, B, Hq, d), dtype=np.float64)
    lses = np.full((num_splits, B, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seqlens[b])
        Kb = gather_paged(k_cache, page_table[b], L, page_size)
        Vb = gather_paged(v_cache, page_table[b], L, page_size)
        for s in range(num_splits):
            lo, hi = bounds[b, s]
            Os[s, b], lses[s, b] = _decode_one(q[b], Kb[lo:hi], Vb[lo:hi], scale, Hq, Hkv)
    return Os, lses


def merge_partials(Os, lses):
    """Combine partial softmaxes: lse = ln sum_s exp(lse_s),
    O = sum_s exp(lse_s - lse) O_s; all-empty gives O = 0, lse = -inf."""
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lses - m_safe[None])             # exp(-inf) = 0 for empty splits
    w = np.where(np.isfinite(lses), w, 0.0)
    Z = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(Z > 0, m_safe + np.log(np.where(Z > 0, Z, 1.0)), -np.inf)
        O = np.where((Z > 0)[..., None], np.sum(w[..., None] * Os, axis=0) / np.where(Z > 0, Z, 1.0)[..., None], 0.0)
    return O, lse


# ----------------------------------------------------------------------------
# Longest-first jagged tile order
# ----------------------------------------------------------------------------

def tile_queue(offsets, heads, causal, kind, tile=128):
    """Work items of the persistent kernels in longest-first order.

    "Optimizing Jagged Flash Attention with TLX", fourth and fifth paragraphs:
    persistent CTAs loop over tiles, and software load balancing of the jagged
    tiles recovers ~20% of the forward. The order used here (a reading; the
    page gives none): items (b, h, t) where t is a query tile (kind="fwd") or
    a key/value tile (kind="bwd") of 128 rows, sorted by descending cost,
    ties by ascending (b, t, h). Cost = number of partner tiles the item
    visits: nt = ceil(L_b / 128) when not causal; t + 1 (fwd) or nt - t (bwd)
    when causal. Returns a list of (b, h, t)."""
    items = []
    for b, (s, e) in enumerate(seq_ranges(offsets)):
        L = e - s
        nt = -(-L // tile)
        for t in range(nt):
            if not causal:
                cost = nt
            elif kind == "fwd":
                cost = t + 1
            else:
                cost = nt - t
            for h in range(heads):
                items.append((-cost, b, t, h))
    items.sort()
    return [(b, h, t) for (_, b, t, h) in items]


# ----------------------------------------------------------------------------
# Varlen attention: separate query / key lengths, grouped-query heads
# ----------------------------------------------------------------------------

def lower_right_visible(Lq, Lk):
    """bool [Lq, Lk]: key j is visible to query i iff j <= i + (Lk - Lq)
    (bottom-right aligned causal mask; equal to the lower triangle when
    Lq == Lk)."""
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    return j <= i + (Lk - Lq)


def _var_scores(Qh, Kh, scale, causal):
    S = scale * (Qh @ Kh.T)
    if causal:
        S = np.where(lower_right_visible(S.shape[0], S.shape[1]), S, -np.inf)
    return S


def _check_heads(q, k):
    Hq, Hkv = q.shape[1], k.shape[1]
    assert Hkv >= 1 and Hq % Hkv == 0, "query heads must be a multiple of KV heads"
    return Hq // Hkv


def varlen_forward(q, k, v, q_offsets, k_offsets, scale, causal=False):
    """Jagged attention with separate query / key packing and grouped heads.

    q [total_q, Hq, d], k and v [total_k, Hkv, d]; q_offsets and k_offsets are
    int [B+1]. Query head h of sequence b attends to KV head h // (Hq / Hkv)
    of the same sequence. Returns O [total_q, Hq, d] and LSE [Hq, total_q];
    a query row with no visible key has O = 0 and LSE = -inf."""
    group = _check_heads(q, k)
    Hq = q.shape[1]
    qr, kr = seq_ranges(q_offsets), seq_ranges(k_offsets)
    assert len(qr) == len(kr), "q_offsets and k_offsets must describe the same batch"
    O = np.zeros((q.shape[0], Hq, v.shape[2]), dtype=np.float64)
    LSE = np.full((Hq, q.shape[0]), -np.inf, dtype=np.float64)
    for (qs, qe), (ks, ke) in zip(qr, kr):
        if qe == qs or ke == ks:
            continue
        for h in range(Hq):
            g = h // group
            S = _var_scores(q[qs:qe, h], k[ks:ke, g], scale, causal)
            P, lse = _softmax_rows(S)
            O[qs:qe, h] = P @ v[ks:ke, g]
            LSE[h, qs:qe] = lse
    return O, LSE


def varlen_backward(q, k, v, do, q_offsets, k_offsets, scale, causal=False):
    """Exact gradient of varlen_forward's O against dO: per (sequence, query
    head) dV = P^T dO, dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D),
    dQ = scale dS K, dK = scale dS^T Q; a KV head's dK and dV are the sums
    over the query heads that read it. Returns dQ [total_q, Hq, d],
    dK and dV [total_k, Hkv, d]."""
    group = _check_heads(q, k)
    Hq = q.shape[1]
    dQ = np.zeros_like(q, dtype=np.float64)
    dK = np.zeros_like(k, dtype=np.float64)
    dV = np.zeros_like(v, dtype=np.float64)
    for (qs, qe), (ks, ke) in zip(seq_ranges(q_offsets), seq_ranges(k_offsets)):
        if qe == qs or ke == ks:
            continue
        for h in range(Hq):
            g = h // group
            Qh, Kh, Vh, dOh = q[qs:qe, h], k[ks:ke, g], v[ks:ke, g], do[qs:qe, h]
            S = _var_scores(Qh, Kh, scale, causal)
            P, _ = _softmax_rows(S)
            O = P @ Vh
            dP = dOh @ Vh.T
            D = np.sum(dOh * O, axis=1)
            dS = P * (dP - D[:, None])
            dQ[qs:qe, h] = scale * (dS @ Kh)
            dK[ks:ke, g] += scale * (dS.T @ Qh)
            dV[ks:ke, g] += P.T @ dOh
    return dQ, dK, dV


def varlen_tile_queue(q_offsets, k_offsets, q_heads, kv_heads, causal, kind, tile=128):
    """Longest-first work order for varlen attention (same rule as tile_queue).

    kind="fwd": items (b, h, t) for query head h and query tile t; cost = the
    key tiles holding at least one key visible to a row of the tile.
    kind="bwd": items (b, g, u) for KV head g and key tile u; cost = (Hq / Hkv)
    x the query tiles holding at least one query that sees a key of the tile.
    Items of cost 0 are kept (their outputs are zero). Sorted by descending
    cost, ties by ascending (b, tile, head). Returns a list of (b, head, tile)."""
    group = q_heads // kv_heads
    items = []
    for b, ((qs, qe), (ks, ke)) in enumerate(zip(seq_ranges(q_offsets), seq_ranges(k_offsets))):
        Lq, Lk = qe - qs, ke - ks
        vis = lower_right_visible(Lq, Lk) if causal else np.ones((Lq, Lk), dtype=bool)
        nq, nk = -(-Lq // tile), -(-Lk // tile)
        if kind == "fwd":
            for t in range(nq):
                cost = sum(bool(vis[t * tile:(t + 1) * tile, u * tile:(u + 1) * tile].any()) for u in range(nk))
                for h in range(q_heads):
                    items.append((-cost, b, t, h))
        else:
            for u in range(nk):
                cost = group * sum(bool(vis[t * tile:(t + 1) * tile, u * tile:(u + 1) * tile].any())
                                   for t in range(nq))
                for g in range(kv_heads):
                    items.append((-cost, b, u, g))
    items.sort()
    return [(b, h, t) for (_, b, t, h) in items]


# ----------------------------------------------------------------------------
# Small-query paged decode: several query tokens per sequence
# ----------------------------------------------------------------------------
#
# "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul), section
# "PR 1993" (tiles sized to few query rows, e.g. speculative decoding), with
# the split-KV (PR 1940), paging (PR 1999 / PR 2104) and GQA packing (PR 2186)
# of the one-token decode. Reading (the page gives no layout): sequence b
# holds L_b tokens in the cache, the last q_len of them are the new queries;
# query i sits at key position L_b - q_len + i and sees keys j <= that
# position (the bottom-right causal reading of varlen_forward).

def split_counts(seqlens, num_splits, min_split_tokens):
    """Per-sequence split count: num_splits, or with min_split_tokens > 0,
    clamp(ceil(L_b / min_split_tokens), 1, num_splits)."""
    out = []
    for L in (int(x) for x in np.asarray(seqlens).reshape(-1)):
        if min_split_tokens > 0:
            out.append(max(1, min(int(num_splits), -(-L // int(min_split_tokens)))))
        else:
            out.append(int(num_splits))
    return np.asarray(out, dtype=np.int64)


def split_bounds_per_seq(seqlens, num_splits, counts):
    """int64 [B, num_splits, 2]: sequence b is split into counts[b] parts with
    c_b = ceil(L_b / counts[b]), part s covering [s c_b, min((s+1) c_b, L_b));
    parts s >= counts[b] (and parts starting at or past L_b) are (L_b, L_b)."""
    seqlens = [int(x) for x in np.asarray(seqlens).reshape(-1)]
    out = np.zeros((len(seqlens), int(num_splits), 2), dtype=np.int64)
    for b, L in enumerate(seqlens):
        Sb = int(counts[b])
        c = -(-L // Sb) if L > 0 else 0
        for s in range(int(num_splits)):
            if s < Sb:
                out[b, s] = (min(s * c, L), min((s + 1) * c, L))
            else:
                out[b, s] = (L, L)
    return out


def _smallq_one(qb, Kb, Vb, scale, causal=True):
    """qb [q_len, Hq, d] against gathered Kb, Vb [L, Hkv, d] of one sequence."""
    ql, L = qb.shape[0], Kb.shape[0]
    return varlen_forward(qb, Kb, Vb, [0, ql], [0, L], scale, causal)


def decode_smallq_forward(q, k_cache, v_cache, page_table, seqlens, page_size, scale, batch_ids=None):
    """Unsplit small-query paged decode. q [B, q_len, Hq, d]; caches
    [num_pages, P, Hkv, d]. Returns O [B, q_len, Hq, d] and LSE [B, q_len, Hq]
    (rows of `batch_ids` only, if given)."""
    B, ql, Hq, d = q.shape
    ids = range(B) if batch_ids is None else batch_ids
    O = np.zeros((B, ql, Hq, d), dtype=np.float64)
    LSE = np.full((B, ql, Hq), -np.inf, dtype=np.float64)
    for b in ids:
        L = int(seqlens[b])
        Kb = gather_paged(k_cache, page_table[b], L, page_size)
        Vb = gather_paged(v_cache, page_table[b], L, page_size)
        if L == 0:
            continue
        Ob, Lb = _smallq_one(q[b], Kb, Vb, scale)
        O[b], LSE[b] = Ob, Lb.T
    return O, LSE


def decode_smallq_split_partials(q, k_cache, v_cache, page_table, seqlens, page_size, scale, num_splits,
                                 min_split_tokens=0):
    """Per-split partials of the small-query decode: O_s [S, B, q_len, Hq, d]
    (normalised within the split) and lse_s [S, B, q_len, Hq] (-inf where the
    split holds no key visible to the row). Keys outside a split are dropped;
    the causal limit of each query row is the unsplit one."""
    B, ql, Hq, d = q.shape
    counts = split_counts(seqlens, num_splits, min_split_tokens)
    bounds = split_bounds_per_seq(seqlens, num_splits, counts)
    Os = np.zeros((num_splits, B, ql, Hq, d), dtype=np.float64)
    lses = np.full((num_splits, B, ql, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(seqlens[b])
        Kb = gather_paged(k_cache, page_table[b], L, page_size)
        Vb = gather_paged(v_cache, page_table[b], L, page_size)
        group = Hq // Kb.shape[1]
        for s in range(num_splits):
            lo, hi = (int(x) for x in bounds[b, s])
            if hi == lo:
                continue
            for i in range(ql):
                pos = L - ql + i  # key position of query i
                for h in range(Hq):
                    keys = [j for j in range(lo, hi) if j <= pos]
                    if not keys:
                        continue
                    Oh, lse, _ = _head_forward(q[b, i, h][None], Kb[keys, h // group], Vb[keys, h // group], scale,
                                               False)
                    Os[s, b, i, h] = Oh[0]
                    lses[s, b, i, h] = lse[0]
    return Os, lses


# ----------------------------------------------------------------------------
# FP8 (e4m3) inputs
# ----------------------------------------------------------------------------
#
# "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul), section
# "PR 2109: Support FP8 Inputs": the forward takes FP8 inputs for inference.
# The page gives neither the FP8 format nor a scale convention. Reading: e4m3
# (the 8-bit format with 4 exponent and 3 mantissa bits, the one with the range
# for activations) with one descale factor per tensor, so an input byte x of
# tensor T stands for e4m3(x) * T_descale. What the forward computes is then
# exact attention over those real values, and the output is bf16.

def e4m3_decode(codes):
    """float64 values of e4m3 byte codes (uint8 array), from the format's
    definition: bit 7 sign, bits 6-3 exponent with bias 7, bits 2-0 mantissa;
    exponent field 0 is subnormal (mantissa / 8 * 2^-6); exponent 15 with
    mantissa 7 is NaN; there are no infinities, so the largest value is 448."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)


def attention_forward_fp8(q8, k8, v8, offsets, scale, causal, q_descale, k_descale, v_descale):
    """Jagged attention over FP8 inputs: q8, k8, v8 are uint8 e4m3 codes
    [total, H, d]; each stands for its decoded value times the tensor's
    descale. Returns O [total, H, d] and LSE [H, total] of exact attention
    over those values (attention_forward on the dequantized tensors)."""
    q = e4m3_decode(q8) * float(q_descale)
    k = e4m3_decode(k8) * float(k_descale)
    v = e4m3_decode(v8) * float(v_descale)
    return attention_forward(q, k, v, offsets, scale, causal)
