"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError when
the oracle disagrees with a closed form, a brute-force computation, finite
differences, a library routine in a special case, or an invariant of the
mathematics. ``test_oracle_pins.py`` runs them on the real oracle (all must
pass) and on mutants with planted mistakes (at least one must fail).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_form_cases.json")

_ENV = {"log": math.log, "exp": math.exp, "e": math.e, "__builtins__": {}}


def _ev(x):
    """Evaluate a hand-written closed-form expression from the golden file."""
    if isinstance(x, list):
        return [_ev(y) for y in x]
    if isinstance(x, (int, float)):
        return float(x)
    return float(eval(x, _ENV))  # expressions use only numbers, log, exp, e


def _arr(x):
    return np.asarray(_ev(x), dtype=np.float64)


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    m = float(np.max(err)) if err.size else 0.0
    assert m <= tol, f"{what}: max|diff| {m:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- closed forms

def pin_golden_attention(o):
    g = golden()
    for name in ("two_keys", "causal_pair"):
        c = g[name]
        q, k, v, do = (_arr(c[x])[:, None, :] for x in ("q", "k", "v", "do"))
        off = np.array([0, q.shape[0]])
        scale = _ev(c["scale"])
        O, LSE = o.attention_forward(q, k, v, off, scale, c["causal"])
        _close(O[:, 0], _arr(c["o"]), 1e-13, f"{name} O")
        _close(LSE[0], _arr(c["lse"]), 1e-13, f"{name} LSE")
        dQ, dK, dV, _ = o.attention_backward(q, k, v, do, off, scale, c["causal"])
        _close(dQ[:, 0], _arr(c["dq"]), 1e-13, f"{name} dQ")
        _close(dK[:, 0], _arr(c["dk"]), 1e-13, f"{name} dK")
        _close(dV[:, 0], _arr(c["dv"]), 1e-13, f"{name} dV")


def pin_golden_decode(o):
    c = golden()["paged_gqa_decode"]
    q = _arr(c["q"])
    kc = _arr(c["k_cache"])
    vc = _arr(c["v_cache"])
    pt = np.asarray(c["page_table"])
    sl = np.asarray(c["seqlens"])
    O, LSE = o.decode_forward(q, kc, vc, pt, sl, c["page_size"], _ev(c["scale"]))
    _close(O, _arr(c["o"]), 1e-12, "decode O")
    _close(LSE, _arr(c["lse"]), 1e-13, "decode LSE")
    for S in (1, 2, 3, 4):
        Os, ls = o.decode_split_partials(q, kc, vc, pt, sl, c["page_size"], _ev(c["scale"]), S)
        O2, L2 = o.merge_partials(Os, ls)
        _close(O2, _arr(c["o"]), 1e-12, f"decode split {S} O")
        _close(L2, _arr(c["lse"]), 1e-13, f"decode split {S} LSE")


def pin_golden_split_bounds(o):
    c = golden()["split_bounds"]
    got = o.split_bounds(np.asarray(c["seqlens"]), c["num_splits"])
    assert got.tolist() == c["bounds"], got.tolist()


# ---------------------------------------------------------------- special cases

def pin_length_one(o):
    """A length-1 sequence returns its own V row and LSE = scale q.k0."""
    r = _rng(1)
    q, k, v = (r.standard_normal((1, 3, 5)) for _ in range(3))
    O, LSE = o.attention_forward(q, k, v, np.array([0, 1]), 0.7, False)
    _close(O, v, 1e-15, "L=1 O")
    _close(LSE[:, 0], 0.7 * np.sum(q[0] * k[0], axis=-1), 1e-14, "L=1 LSE")


def pin_constant_v(o):
    """If every V row equals the same vector, O equals that vector."""
    r = _rng(2)
    L = 9
    q, k = r.standard_normal((L, 2, 4)), r.standard_normal((L, 2, 4))
    row = r.standard_normal((1, 2, 4))
    v = np.repeat(row, L, axis=0)
    for causal in (False, True):
        O, _ = o.attention_forward(q, k, v, np.array([0, L]), 0.5, causal)
        _close(O, v, 1e-13, f"constant V (causal={causal})")


def pin_rows_sum_to_one(o):
    """With V = identity (d_v = L), O equals P itself: rows must sum to 1,
    be non-negative, and be zero on causally hidden keys."""
    r = _rng(3)
    L = 7
    q, k = r.standard_normal((L, 1, 3)), r.standard_normal((L, 1, 3))
    v = np.eye(L)[:, None, :]
    for causal in (False, True):
        P, _ = o.attention_forward(q, k, v, np.array([0, L]), 1.3, causal)
        P = P[:, 0, :]
        _close(P.sum(axis=1), np.ones(L), 1e-14, "row sums")
        assert np.all(P >= 0)
        if causal:
            assert np.all(P[np.triu_indices(L, 1)] == 0.0)


def pin_brute_force_forward(o):
    """Pure-Python loops, softmax by its definition exp(s)/sum exp(s)."""
    r = _rng(4)
    lengths = [3, 1, 5]
    H, d = 2, 3
    off = np.concatenate([[0], np.cumsum(lengths)])
    T = off[-1]
    q, k, v = (r.standard_normal((T, H, d)) for _ in range(3))
    scale = 0.9
    for causal in (False, True):
        O, LSE = o.attention_forward(q, k, v, off, scale, causal)
        for b in range(len(lengths)):
            s0, s1 = off[b], off[b + 1]
            for h in range(H):
                for i in range(s0, s1):
                    js = [j for j in range(s0, s1) if (not causal or j - s0 <= i - s0)]
                    sc = [scale * sum(q[i, h, x] * k[j, h, x] for x in range(d)) for j in js]
                    z = sum(math.exp(t) for t in sc)
                    for x in range(d):
                        ref = sum(math.exp(t) / z * v[j, h, x] for t, j in zip(sc, js))
                        assert abs(O[i, h, x] - ref) < 1e-12, (b, h, i, x)
                    assert abs(LSE[h, i] - math.log(z)) < 1e-12


def _loss(o, q, k, v, do, off, scale, causal):
    O, _ = o.attention_forward(q, k, v, off, scale, causal)
    return float(np.sum(O * do))


def pin_finite_differences(o):
    """Analytic gradients of sum(dO*O) against central differences, h = 1e-6."""
    r = _rng(5)
    lengths = [2, 4]
    H, d = 2, 3
    off = np.concatenate([[0], np.cumsum(lengths)])
    T = off[-1]
    scale = 0.8
    for causal in (False, True):
        q, k, v, do = (r.standard_normal((T, H, d)) for _ in range(4))
        dQ, dK, dV, _ = o.attention_backward(q, k, v, do, off, scale, causal)
        for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + 1e-6
                fp = _loss(o, q, k, v, do, off, scale, causal)
                x[idx] = old - 1e-6
                fm = _loss(o, q, k, v, do, off, scale, causal)
                x[idx] = old
                num[idx] = (fp - fm) / 2e-6
            rel = np.max(np.abs(num - g)) / max(np.max(np.abs(g)), 1e-30)
            assert rel < 1e-6, f"d{name} (causal={causal}) rel err {rel:.2e}"


def pin_torch_sdpa(o):
    """torch's fp64 CPU scaled_dot_product_attention (forward) and autograd
    (backward), applied per sequence, as a library special case."""
    r = _rng(6)
    lengths = [5, 1, 8, 3]
    H, d = 3, 4
    off = np.concatenate([[0], np.cumsum(lengths)])
    T = off[-1]
    scale = 0.6
    for causal in (False, True):
        q, k, v, do = (r.standard_normal((T, H, d)) for _ in range(4))
        O, LSE = o.attention_forward(q, k, v, off, scale, causal)
        dQ, dK, dV, _ = o.attention_backward(q, k, v, do, off, scale, causal)
        for b in range(len(lengths)):
            s0, s1 = off[b], off[b + 1]
            tq, tk, tv = (torch.tensor(x[s0:s1].transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
            out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale, is_causal=causal)
            out.backward(torch.tensor(do[s0:s1].transpose(1, 0, 2)))
            _close(O[s0:s1], out.detach().numpy().transpose(1, 0, 2), 1e-12, "sdpa O")
            _close(dQ[s0:s1], tq.grad.numpy().transpose(1, 0, 2), 1e-12, "autograd dQ")
            _close(dK[s0:s1], tk.grad.numpy().transpose(1, 0, 2), 1e-12, "autograd dK")
            _close(dV[s0:s1], tv.grad.numpy().transpose(1, 0, 2), 1e-12, "autograd dV")
            # LSE from the scores via torch.logsumexp
            S = scale * torch.einsum("hid,hjd->hij", tq.detach(), tk.detach())
            if causal:
                L = s1 - s0
                S = S.masked_fill(~torch.tril(torch.ones(L, L, dtype=torch.bool)), float("-inf"))
            _close(LSE[:, s0:s1], torch.logsumexp(S, dim=-1).numpy(), 1e-12, "logsumexp")


def pin_jagged_equals_separate(o):
    """Packing is transparent: each sequence's result equals attention on that
    sequence alone, whatever its neighbours are."""
    r = _rng(7)
    lengths = [4, 0, 6, 2]
    H, d = 2, 3
    off = np.concatenate([[0], np.cumsum(lengths)])
    T = off[-1]
    q, k, v, do = (r.standard_normal((T, H, d)) for _ in range(4))
    O, LSE = o.attention_forward(q, k, v, off, 1.1, False)
    dQ, dK, dV, D = o.attention_backward(q, k, v, do, off, 1.1, False)
    for b in range(len(lengths)):
        s0, s1 = off[b], off[b + 1]
        if s0 == s1:
            continue
        one = np.array([0, s1 - s0])
        O1, L1 = o.attention_forward(q[s0:s1], k[s0:s1], v[s0:s1], one, 1.1, False)
        g1 = o.attention_backward(q[s0:s1], k[s0:s1], v[s0:s1], do[s0:s1], one, 1.1, False)
        _close(O[s0:s1], O1, 0.0, "packed O")
        _close(LSE[:, s0:s1], L1, 0.0, "packed LSE")
        for a, bb in zip((dQ, dK, dV), g1[:3]):
            _close(a[s0:s1], bb, 0.0, "packed grads")


def pin_delta_identity(o):
    """D = rowsum(dO * O) equals rowsum(P * dP) with dP = dO V^T."""
    r = _rng(8)
    L, d = 6, 4
    q, k, v, do = (r.standard_normal((L, 1, d)) for _ in range(4))
    off = np.array([0, L])
    _, _, _, D = o.attention_backward(q, k, v, do, off, 0.5, False)
    P, _ = o.attention_forward(q, k, np.eye(L)[:, None, :], off, 0.5, False)
    dP = do[:, 0] @ v[:, 0].T
    _close(D[0], np.sum(P[:, 0] * dP, axis=1), 1e-13, "delta identity")


def pin_broadcast(o):
    """Broadcast-Q equals per-sequence attention with a copy of Q, and its dQ
    equals the sum over the batch of those per-sequence dQ (torch autograd)."""
    r = _rng(9)
    lengths = [3, 7, 1]
    Lq, H, d = 4, 2, 3
    off = np.concatenate([[0], np.cumsum(lengths)])
    T = off[-1]
    q = r.standard_normal((Lq, H, d))
    k, v = r.standard_normal((T, H, d)), r.standard_normal((T, H, d))
    do = r.standard_normal((len(lengths), Lq, H, d))
    scale = 0.7
    O, LSE = o.broadcast_forward(q, k, v, off, scale)
    dQ, dK, dV = o.broadcast_backward(q, k, v, do, off, scale)
    tq = torch.tensor(q.transpose(1, 0, 2), requires_grad=True)
    for b in range(len(lengths)):
        s0, s1 = off[b], off[b + 1]
        tk = torch.tensor(k[s0:s1].transpose(1, 0, 2), requires_grad=True)
        tv = torch.tensor(v[s0:s1].transpose(1, 0, 2), requires_grad=True)
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
        out.backward(torch.tensor(do[b].transpose(1, 0, 2)))
        _close(O[b], out.detach().numpy().transpose(1, 0, 2), 1e-12, "bcast O")
        _close(dK[s0:s1], tk.grad.numpy().transpose(1, 0, 2), 1e-12, "bcast dK")
        _close(dV[s0:s1], tv.grad.numpy().transpose(1, 0, 2), 1e-12, "bcast dV")
        S = scale * torch.einsum("hid,hjd->hij", tq.detach(), tk.detach())
        _close(LSE[b], torch.logsumexp(S, -1).numpy(), 1e-12, "bcast LSE")
    _close(dQ, tq.grad.numpy().transpose(1, 0, 2), 1e-12, "bcast dQ = sum over batch")


def _random_paged(r, lengths, Hq, Hkv, d, P):
    pages = [-(-L // P) for L in lengths]
    n = max(sum(pages), 1)
    perm = r.permutation(n)
    pt = np.zeros((len(lengths), max(max(pages), 1)), dtype=np.int64)
    c = 0
    for b, m in enumerate(pages):
        pt[b, :m] = perm[c:c + m]
        c += m
    q = r.standard_normal((len(lengths), Hq, d))
    kc = r.standard_normal((n, P, Hkv, d))
    vc = r.standard_normal((n, P, Hkv, d))
    return q, kc, vc, pt


def pin_decode(o):
    """Paged GQA decode equals torch SDPA on the gathered dense K/V with each
    query head attending its KV group; split+merge equals unsplit; the result
    does not depend on where the pages sit."""
    r = _rng(10)
    lengths = np.array([5, 1, 0, 13, 8])
    Hq, Hkv, d = 6, 2, 4
    scale = 0.45
    for P in (1, 3, 16):
        q, kc, vc, pt = _random_paged(r, lengths, Hq, Hkv, d, P)
        O, LSE = o.decode_forward(q, kc, vc, pt, lengths, P, scale)
        for b, L in enumerate(lengths):
            if L == 0:
                assert np.all(O[b] == 0) and np.all(np.isneginf(LSE[b]))
                continue
            Kd = np.stack([kc[pt[b, t // P], t % P] for t in range(L)])    # [L, Hkv, d]
            Vd = np.stack([vc[pt[b, t // P], t % P] for t in range(L)])
            grp = Hq // Hkv
            tk = torch.tensor(np.repeat(Kd, grp, axis=1).transpose(1, 0, 2))
            tv = torch.tensor(np.repeat(Vd, grp, axis=1).transpose(1, 0, 2))
            tq = torch.tensor(q[b][:, None, :])
            ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[:, 0]
            _close(O[b], ref.numpy(), 1e-12, f"decode P={P}")
            S = scale * torch.einsum("hd,hjd->hj", tq[:, 0], tk)
            _close(LSE[b], torch.logsumexp(S, -1).numpy(), 1e-12, "decode LSE")
        for S_ in (1, 2, 5, 16):
            Os, ls = o.decode_split_partials(q, kc, vc, pt, lengths, P, scale, S_)
            O2, L2 = o.merge_partials(Os, ls)
            _close(O2, O, 1e-12, f"split {S_} O")
            _close(L2, LSE, 1e-12, f"split {S_} LSE")
        # moving every page elsewhere (and the table with it) changes nothing
        n = kc.shape[0]
        perm = r.permutation(n)
        kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
        kc2[perm], vc2[perm] = kc, vc
        O3, L3 = o.decode_forward(q, kc2, vc2, perm[pt], lengths, P, scale)
        _close(O3, O, 0.0, "page permutation")
        _close(L3, LSE, 0.0, "page permutation LSE")


def pin_split_cover(o):
    """Every token lies in exactly one split, splits are contiguous and in
    order, and none is longer than ceil(L / S)."""
    for L in (0, 1, 2, 7, 64, 1000, 32768):
        for S in (1, 2, 3, 7, 16, 64):
            bnd = o.split_bounds(np.array([L]), S)[0]
            cover = np.zeros(L, dtype=int)
            prev = 0
            c = -(-L // S)
            for lo, hi in bnd:
                assert lo == prev or lo == hi == L
                assert 0 <= hi - lo <= c
                cover[lo:hi] += 1
                prev = hi
            assert np.all(cover == 1) and prev == L


def pin_tile_queue(o):
    """Every (b, h, tile) appears once; costs never increase; ties go by
    ascending (b, tile, h). Costs are recounted here by brute force: the number
    of partner tiles with at least one visible (query, key) pair."""
    off = np.array([0, 300, 300, 301, 700, 1000])
    H, T = 2, 128
    for causal in (False, True):
        for kind in ("fwd", "bwd"):
            q = o.tile_queue(off, H, causal, kind, T)
            expect = set()
            for b in range(len(off) - 1):
                L = off[b + 1] - off[b]
                for t in range(-(-L // T)):
                    for h in range(H):
                        expect.add((b, h, t))
            assert len(q) == len(expect) and set(q) == expect

            def cost(item):
                b, h, t = item
                L = int(off[b + 1] - off[b])
                n = 0
                for u in range(-(-L // T)):
                    qi, kj = (t, u) if kind == "fwd" else (u, t)
                    rows = range(qi * T, min(qi * T + T, L))
                    cols = range(kj * T, min(kj * T + T, L))
                    if any((not causal) or c <= r_ for r_ in rows for c in cols):
                        n += 1
                return n
            keys = [(-cost(it), it[0], it[2], it[1]) for it in q]
            assert keys == sorted(keys), (causal, kind)



# ---------------------------------------------------------------- varlen / GQA

def _lower_right_library(Lq, Lk):
    """torch's own bottom-right causal mask (torch.nn.attention.bias)."""
    import warnings

    from torch.nn.attention.bias import causal_lower_right
    with warnings.catch_warnings():  # torch warns about SDPA on L_q > L_k; only the mask is used here
        warnings.simplefilter("ignore")
        return causal_lower_right(Lq, Lk)._materialize(device=torch.device("cpu"))


def pin_varlen_torch_lower_right(o):
    """torch fp64 SDPA with torch's lower-right causal mask (or no mask), K/V
    heads expanded by repeat_interleave, and autograd through that expansion
    (which sums dK/dV over a group): a library special case per sequence.
    Every query row here sees at least one key."""
    r = _rng(21)
    q_lens, k_lens = [3, 5, 1, 8], [7, 5, 4, 9]
    Hq, Hkv, d = 4, 2, 3
    qo = np.concatenate([[0], np.cumsum(q_lens)])
    ko = np.concatenate([[0], np.cumsum(k_lens)])
    scale = 0.7
    for causal in (False, True):
        q, do = r.standard_normal((qo[-1], Hq, d)), r.standard_normal((qo[-1], Hq, d))
        k, v = r.standard_normal((ko[-1], Hkv, d)), r.standard_normal((ko[-1], Hkv, d))
        O, LSE = o.varlen_forward(q, k, v, qo, ko, scale, causal)
        dQ, dK, dV = o.varlen_backward(q, k, v, do, qo, ko, scale, causal)
        for b in range(len(q_lens)):
            q0, q1, k0, k1 = qo[b], qo[b + 1], ko[b], ko[b + 1]
            tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True)
                          for x in (q[q0:q1], k[k0:k1], v[k0:k1]))
            ek, ev = (t.repeat_interleave(Hq // Hkv, dim=0) for t in (tk, tv))
            mask = _lower_right_library(q1 - q0, k1 - k0) if causal else None
            out = torch.nn.functional.scaled_dot_product_attention(tq, ek, ev, attn_mask=mask, scale=scale)
            out.backward(torch.tensor(do[q0:q1].transpose(1, 0, 2)))
            _close(O[q0:q1], out.detach().numpy().transpose(1, 0, 2), 1e-12, "varlen sdpa O")
            _close(dQ[q0:q1], tq.grad.numpy().transpose(1, 0, 2), 1e-12, "varlen autograd dQ")
            _close(dK[k0:k1], tk.grad.numpy().transpose(1, 0, 2), 1e-12, "varlen autograd dK")
            _close(dV[k0:k1], tv.grad.numpy().transpose(1, 0, 2), 1e-12, "varlen autograd dV")
            S = scale * torch.einsum("hid,hjd->hij", tq.detach(), ek.detach())
            if causal:
                S = S.masked_fill(~mask, float("-inf"))
            _close(LSE[:, q0:q1], torch.logsumexp(S, dim=-1).numpy(), 1e-12, "varlen logsumexp")


def pin_varlen_brute_force(o):
    """Pure-Python loops with the visibility rule of a query block that ends
    where the keys end (query i of L_q sits at key position i + L_k - L_q),
    including L_q > L_k, where the first L_q - L_k rows see nothing
    (O = 0, LSE = -inf)."""
    r = _rng(22)
    q_lens, k_lens = [5, 2, 3], [2, 6, 0]
    Hq, Hkv, d = 3, 1, 2
    qo = np.concatenate([[0], np.cumsum(q_lens)])
    ko = np.concatenate([[0], np.cumsum(k_lens)])
    q = r.standard_normal((qo[-1], Hq, d))
    k, v = r.standard_normal((ko[-1], Hkv, d)), r.standard_normal((ko[-1], Hkv, d))
    for causal in (False, True):
        O, LSE = o.varlen_forward(q, k, v, qo, ko, 0.9, causal)
        for b in range(len(q_lens)):
            Lq, Lk = q_lens[b], k_lens[b]
            for h in range(Hq):
                for i in range(Lq):
                    pos = i + Lk - Lq  # the query's position on the key axis
                    keys = [j for j in range(Lk) if (not causal) or j <= pos]
                    qi = q[qo[b] + i, h]
                    if not keys:
                        assert np.all(O[qo[b] + i, h] == 0.0) and LSE[h, qo[b] + i] == -np.inf
                        continue
                    s = [0.9 * sum(qi[c] * k[ko[b] + j, 0, c] for c in range(d)) for j in keys]
                    z = sum(math.exp(x) for x in s)
                    out = [sum(math.exp(s[n]) / z * v[ko[b] + j, 0, c] for n, j in enumerate(keys))
                           for c in range(d)]
                    _close(O[qo[b] + i, h], out, 1e-13, "varlen brute-force O")
                    _close(LSE[h, qo[b] + i], math.log(z), 1e-13, "varlen brute-force LSE")


def pin_varlen_finite_differences(o):
    """Central differences (h = 1e-6) of sum(O * dO) for a grouped, bottom-right
    causal case with L_q != L_k: the gradient of a KV head must collect every
    query head of its group."""
    r = _rng(23)
    q_lens, k_lens = [2, 4], [3, 2]
    Hq, Hkv, d = 4, 2, 2
    qo = np.concatenate([[0], np.cumsum(q_lens)])
    ko = np.concatenate([[0], np.cumsum(k_lens)])
    q, do = r.standard_normal((qo[-1], Hq, d)), r.standard_normal((qo[-1], Hq, d))
    k, v = r.standard_normal((ko[-1], Hkv, d)), r.standard_normal((ko[-1], Hkv, d))

    def loss():
        O, _ = o.varlen_forward(q, k, v, qo, ko, 0.8, True)
        return float(np.sum(O * do))
    grads = o.varlen_backward(q, k, v, do, qo, ko, 0.8, True)
    for name, x, g in (("q", q, grads[0]), ("k", k, grads[1]), ("v", v, grads[2])):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + 1e-6
            fp = loss()
            x[idx] = old - 1e-6
            fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / 2e-6
        rel = np.max(np.abs(num - g)) / max(np.max(np.abs(g)), 1e-30)
        assert rel < 1e-6, f"varlen d{name} rel err {rel:.2e}"


def pin_varlen_reduces_to_self(o):
    """With q_offsets == k_offsets and Hkv == Hq, varlen attention is jagged
    self-attention (top-left and bottom-right masks coincide when L_q == L_k)."""
    r = _rng(24)
    lengths = [4, 0, 7, 1]
    off = np.concatenate([[0], np.cumsum(lengths)])
    q, k, v, do = (r.standard_normal((off[-1], 2, 3)) for _ in range(4))
    for causal in (False, True):
        O1, L1 = o.attention_forward(q, k, v, off, 0.6, causal)
        O2, L2 = o.varlen_forward(q, k, v, off, off, 0.6, causal)
        _close(O2, O1, 1e-14, "varlen self O")
        _close(L2, L1, 1e-14, "varlen self LSE")
        g1 = o.attention_backward(q, k, v, do, off, 0.6, causal)
        g2 = o.varlen_backward(q, k, v, do, off, off, 0.6, causal)
        for a, b_ in zip(g2, g1[:3]):
            _close(a, b_, 1e-14, "varlen self grads")


def pin_varlen_tile_queue(o):
    """Every item appears once; costs never increase; ties go by ascending
    (b, tile, head); each cost is recounted from torch's lower-right mask,
    max-pooled over 128 x 128 blocks (a block counts when it holds any
    visible pair)."""
    qo = np.array([0, 300, 300, 301, 700, 1000, 1100])
    ko = np.array([0, 100, 400, 700, 700, 1300, 1350])
    Hq, Hkv, T = 4, 2, 128
    for causal in (False, True):
        for kind in ("fwd", "bwd"):
            got = o.varlen_tile_queue(qo, ko, Hq, Hkv, causal, kind, T)
            heads = Hq if kind == "fwd" else Hkv
            expect_cost = {}
            for b in range(len(qo) - 1):
                Lq, Lk = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
                nq, nk = -(-Lq // T), -(-Lk // T)
                if Lq and Lk:
                    m = _lower_right_library(Lq, Lk) if causal else torch.ones(Lq, Lk, dtype=torch.bool)
                    blocks = torch.nn.functional.max_pool2d(m[None, None].double(), T, T, ceil_mode=True)[0, 0] > 0
                else:
                    blocks = torch.zeros(nq, nk, dtype=torch.bool)
                for t in range(nq if kind == "fwd" else nk):
                    c = int(blocks[t].sum()) if kind == "fwd" else (Hq // Hkv) * int(blocks[:, t].sum())
                    for h in range(heads):
                        expect_cost[(b, h, t)] = c
            assert len(got) == len(expect_cost) and set(got) == set(expect_cost), (causal, kind)
            keys = [(-expect_cost[it], it[0], it[2], it[1]) for it in got]
            assert keys == sorted(keys), (causal, kind)



# ---------------------------------------------------------------- small-query paged decode

def pin_golden_smallq_decode(o):
    c = golden()["smallq_paged_decode"]
    args = (_arr(c["q"]), _arr(c["k_cache"]), _arr(c["v_cache"]), np.asarray(c["page_table"]),
            np.asarray(c["seqlens"]), c["page_size"], _ev(c["scale"]))
    O, LSE = o.decode_smallq_forward(*args)
    _close(O, _arr(c["o"]), 1e-13, "small-query decode O")
    _close(LSE, _arr(c["lse"]), 1e-13, "small-query decode LSE")
    for S in (1, 2, 3):
        Os, ls = o.decode_smallq_split_partials(*args, S)
        O2, L2 = o.merge_partials(Os, ls)
        _close(O2, _arr(c["o"]), 1e-13, f"small-query split {S} O")
        _close(L2, _arr(c["lse"]), 1e-13, f"small-query split {S} LSE")


def pin_golden_dynamic_split_counts(o):
    c = golden()["dynamic_split_counts"]
    got = o.split_counts(np.asarray(c["seqlens"]), c["num_splits"], c["min_split_tokens"])
    assert got.tolist() == c["counts"], got.tolist()
    b = o.split_bounds_per_seq([1000], 6, [4])[0]
    assert b.tolist() == c["bounds_1000_of_6"], b.tolist()
    # without a minimum every sequence takes num_splits parts (the one-token decode rule)
    assert o.split_counts([5, 0, 99], 7, 0).tolist() == [7, 7, 7]
    assert (o.split_bounds_per_seq([10, 2, 0], 4, [4, 4, 4]) == o.split_bounds([10, 2, 0], 4)).all()


def pin_smallq_brute_force(o):
    """Pure-Python loops: gather each token through the page table by hand,
    query i of q_len sits at key position L - q_len + i."""
    r = _rng(41)
    lengths, ql, Hq, Hkv, d, P = [5, 2, 7], 3, 4, 2, 2, 3
    _, kc, vc, pt = _random_paged(r, lengths, Hq, Hkv, d, P)
    q = r.standard_normal((len(lengths), ql, Hq, d))
    O, LSE = o.decode_smallq_forward(q, kc, vc, pt, np.array(lengths), P, 0.8)
    for b, L in enumerate(lengths):
        for i in range(ql):
            pos = L - ql + i
            for h in range(Hq):
                g = h // (Hq // Hkv)
                keys = [j for j in range(L) if j <= pos]
                if not keys:
                    assert np.all(O[b, i, h] == 0.0) and LSE[b, i, h] == -np.inf
                    continue
                rows_k = [kc[int(pt[b][j // P]), j % P, g] for j in keys]
                rows_v = [vc[int(pt[b][j // P]), j % P, g] for j in keys]
                sc = [0.8 * sum(q[b, i, h, c] * kr[c] for c in range(d)) for kr in rows_k]
                z = sum(math.exp(x) for x in sc)
                out = [sum(math.exp(sc[n]) / z * rows_v[n][c] for n in range(len(keys))) for c in range(d)]
                _close(O[b, i, h], out, 1e-13, "small-query brute-force O")
                _close(LSE[b, i, h], math.log(z), 1e-13, "small-query brute-force LSE")


def pin_smallq_reduces_to_decode(o):
    """One query token per sequence is the one-token paged decode."""
    r = _rng(42)
    lengths, Hq, Hkv, d, P = [9, 1, 0, 17], 8, 2, 4, 4
    _, kc, vc, pt = _random_paged(r, lengths, Hq, Hkv, d, P)
    q = r.standard_normal((len(lengths), 1, Hq, d))
    O, LSE = o.decode_smallq_forward(q, kc, vc, pt, np.array(lengths), P, 0.5)
    O1, L1 = o.decode_forward(q[:, 0], kc, vc, pt, np.array(lengths), P, 0.5)
    _close(O[:, 0], O1, 1e-14, "q_len 1 O")
    _close(LSE[:, 0], L1, 1e-14, "q_len 1 LSE")


def pin_smallq_split_merge(o):
    """Splits with per-sequence counts, merged, equal the unsplit result."""
    r = _rng(43)
    lengths, ql, Hq, Hkv, d, P = [40, 3, 1, 0, 25], 4, 4, 1, 3, 5
    _, kc, vc, pt = _random_paged(r, lengths, Hq, Hkv, d, P)
    q = r.standard_normal((len(lengths), ql, Hq, d))
    O, LSE = o.decode_smallq_forward(q, kc, vc, pt, np.array(lengths), P, 0.7)
    for S, mn in ((1, 0), (3, 0), (8, 0), (8, 10), (5, 7)):
        Os, ls = o.decode_smallq_split_partials(q, kc, vc, pt, np.array(lengths), P, 0.7, S, mn)
        O2, L2 = o.merge_partials(Os, ls)
        _close(O2, O, 1e-12, f"small-query split {S}/{mn} O")
        _close(L2, LSE, 1e-12, f"small-query split {S}/{mn} LSE")



# ---------------------------------------------------------------- FP8 inputs

def pin_e4m3_decode(o):
    """The e4m3 decoder against hand-derived codes and against torch's own
    float8_e4m3fn type for all 256 codes (NaN where torch has NaN)."""
    hand = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0,
            0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5}
    for code, val in hand.items():
        got = float(o.e4m3_decode(np.array([code], dtype=np.uint8))[0])
        assert got == val, (hex(code), got, val)
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = o.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def pin_fp8_attention(o):
    """FP8 attention is attention over the dequantized inputs; with unit
    descales and inputs that are already e4m3 values it equals torch fp64 SDPA."""
    r = _rng(51)
    lengths = [5, 1, 9]
    off = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d = off[-1], 2, 4
    x = [torch.tensor(r.standard_normal((T, H, d))).to(torch.float8_e4m3fn) for _ in range(3)]
    codes = [t.view(torch.uint8).numpy() for t in x]
    for causal in (False, True):
        O, LSE = o.attention_forward_fp8(*codes, off, 0.5, causal, 1.0, 1.0, 1.0)
        for b in range(len(lengths)):
            s0, s1 = off[b], off[b + 1]
            tq, tk, tv = (t[s0:s1].to(torch.float64).transpose(0, 1) for t in x)
            ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.5, is_causal=causal)
            _close(O[s0:s1], ref.numpy().transpose(1, 0, 2), 1e-12, "fp8 attention vs sdpa")
    # descales: scaling K by c is scaling the softmax scale by c; scaling V scales O
    O1, L1 = o.attention_forward_fp8(*codes, off, 0.5, False, 1.0, 2.0, 3.0)
    O2, L2 = o.attention_forward_fp8(*codes, off, 1.0, False, 1.0, 1.0, 1.0)
    _close(O1, 3.0 * O2, 1e-12, "fp8 descales O")
    _close(L1, L2, 1e-12, "fp8 descales LSE")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
