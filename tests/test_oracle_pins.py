"""The oracle against its pins, and planted mistakes against the same pins.

No GPU needed. A pin is something other than the oracle itself: a
hand-derived closed form, brute force in plain loops, central finite
differences, torch's fp64 attention/autograd in a special case, or an
invariant. The mutation tests plant plausible mistakes in a copy of the
oracle (on the CPU) and require that at least one pin catches each.
"""
import importlib

import numpy as np
import pytest

import oracle.attention as real_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(real_oracle)


def _mutant(patch):
    """A fresh copy of the oracle module with one function replaced."""
    spec = importlib.util.find_spec("oracle.attention")
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    patch(m)
    return m


def _bwd_variant(kind):
    def make(m):
        orig_scores = m._scores
        orig_soft = m._softmax_rows

        def hb(Qh, Kh, Vh, dOh, scale, causal):
            S = orig_scores(Qh, Kh, scale, causal)
            P, _ = orig_soft(S)
            O = P @ Vh
            dV = P.T @ dOh
            dP = dOh @ Vh.T
            D = np.sum(dOh * O, axis=1)
            if kind == "drop_delta":
                dS = P * dP
            elif kind == "sign_dS":
                dS = P * (D[:, None] - dP)
            else:
                dS = P * (dP - D[:, None])
            dQ = scale * (dS @ Kh)
            dK = scale * (dS.T @ Qh)
            if kind == "dq_no_scale":
                dQ = dS @ Kh
            if kind == "dk_no_scale":
                dK = dS.T @ Qh
            if kind == "dv_transposed":
                dV = (P @ dOh) if P.shape[0] == P.shape[1] else P.T @ dOh * 1.01
            return dQ, dK, dV, D
        m._head_backward = hb
    return make


def _fwd_variant(kind):
    def make(m):
        orig = m._scores

        def sc(Qh, Kh, scale, causal):
            if kind == "no_scale":
                return orig(Qh, Kh, 1.0, causal)
            if kind == "causal_upper":
                S = scale * (Qh @ Kh.T)
                if causal:
                    L = S.shape[0]
                    S = np.where(np.triu(np.ones((L, L), dtype=bool)), S, -np.inf)
                return S
            return orig(Qh, Kh, scale, causal)
        m._scores = sc
    return make


def _lse_log2(m):
    orig = m._softmax_rows

    def soft(S):
        P, lse = orig(S)
        return P, lse / np.log(2.0)
    m._softmax_rows = soft


def _merge_no_reweight(m):
    def merge(Os, lses):
        O, lse = real_oracle.merge_partials(Os, lses)
        valid = np.isfinite(lses).sum(axis=0)
        Oavg = np.where((valid > 0)[..., None], np.sum(np.where(np.isfinite(lses)[..., None], Os, 0.0), 0) / np.maximum(valid, 1)[..., None], 0.0)
        return Oavg, lse
    m.merge_partials = merge


def _gqa_wrong_group(m):
    orig = m._decode_one

    def one(qb, Kb, Vb, scale, q_heads, kv_heads):
        # maps query head h to KV head h % Hkv instead of h // (Hq / Hkv)
        O, L = orig(qb, Kb, Vb, scale, q_heads, kv_heads)
        group = q_heads // kv_heads
        if Kb.shape[0] and group > 1:
            for h in range(q_heads):
                g = h % kv_heads
                Oh, lse, _ = m._head_forward(qb[h:h + 1], Kb[:, g], Vb[:, g], scale, False)
                O[h], L[h] = Oh[0], lse[0]
        return O, L
    m._decode_one = one


def _page_slot_off_by_one(m):
    def gather(cache, row, length, P):
        idx_page = np.asarray([int(row[t // P]) for t in range(length)], dtype=np.int64)
        idx_slot = (np.arange(length) + (1 if P > 1 else 0)) % P
        return cache[idx_page, idx_slot]
    m.gather_paged = gather


def _queue_ascending(m):
    orig = m.tile_queue

    def q(*a, **k):
        return list(reversed(orig(*a, **k)))
    m.tile_queue = q


def _varlen_top_left(m):
    # aligns the varlen causal mask to the top left (j <= i) instead of the bottom right
    def vis(Lq, Lk):
        return np.arange(Lk)[None, :] <= np.arange(Lq)[:, None]
    m.lower_right_visible = vis


def _varlen_gqa_modulo(m):
    # query head h reads KV head h % Hkv instead of h // (Hq / Hkv)
    def fwd(q, k, v, qo, ko, scale, causal=False):
        Hq, Hkv = q.shape[1], k.shape[1]
        perm = [h % Hkv for h in range(Hq)]
        kk = k[:, perm]
        vv = v[:, perm]
        return real_oracle.varlen_forward(q, kk, vv, qo, ko, scale, causal)
    m.varlen_forward = fwd


def _varlen_dk_last_head(m):
    # a KV head's dK keeps only the last query head of its group
    def bwd(q, k, v, do, qo, ko, scale, causal=False):
        Hq, Hkv = q.shape[1], k.shape[1]
        G = Hq // Hkv
        dQ, dK, dV = real_oracle.varlen_backward(q, k, v, do, qo, ko, scale, causal)
        kk = np.repeat(k, G, axis=1)
        vv = np.repeat(v, G, axis=1)
        _, dK1, _ = real_oracle.varlen_backward(q, kk, vv, do, qo, ko, scale, causal)
        return dQ, dK1[:, G - 1::G], dV
    m.varlen_backward = bwd


def _smallq_top_left(m):
    # query i of the small-query decode sees keys 0..i (its position counted from the start)
    def one(qb, Kb, Vb, scale, causal=True):
        ql, L = qb.shape[0], Kb.shape[0]
        if ql <= L:
            O, lse = real_oracle.varlen_forward(qb, Kb[:ql], Vb[:ql], [0, ql], [0, ql], scale, True)
            return O, lse
        return real_oracle.varlen_forward(qb, Kb, Vb, [0, ql], [0, L], scale, causal)
    m._smallq_one = one


def _split_counts_floor(m):
    # floor instead of ceiling in the per-sequence split count
    def counts(seqlens, num_splits, min_split_tokens):
        out = []
        for L in (int(x) for x in np.asarray(seqlens).reshape(-1)):
            out.append(max(1, min(num_splits, L // min_split_tokens)) if min_split_tokens > 0 else num_splits)
        return np.asarray(out, dtype=np.int64)
    m.split_counts = counts


def _e4m3_bias_8(m):
    # exponent bias 8 instead of 7
    orig = m.e4m3_decode

    def dec(codes):
        return orig(codes) * 0.5
    m.e4m3_decode = dec


def _fp8_no_v_descale(m):
    def fwd(q8, k8, v8, offsets, scale, causal, qd, kd, vd):
        return real_oracle.attention_forward_fp8(q8, k8, v8, offsets, scale, causal, qd, kd, 1.0)
    m.attention_forward_fp8 = fwd


MUTANTS = {
    "bwd_drop_delta": _bwd_variant("drop_delta"),
    "bwd_sign_dS": _bwd_variant("sign_dS"),
    "bwd_dq_no_scale": _bwd_variant("dq_no_scale"),
    "bwd_dk_no_scale": _bwd_variant("dk_no_scale"),
    "bwd_dv_transposed": _bwd_variant("dv_transposed"),
    "fwd_no_scale": _fwd_variant("no_scale"),
    "fwd_causal_upper": _fwd_variant("causal_upper"),
    "lse_in_log2": _lse_log2,
    "merge_no_reweight": _merge_no_reweight,
    "gqa_wrong_group": _gqa_wrong_group,
    "page_slot_off_by_one": _page_slot_off_by_one,
    "queue_ascending": _queue_ascending,
    "varlen_top_left": _varlen_top_left,
    "varlen_gqa_modulo": _varlen_gqa_modulo,
    "varlen_dk_last_head": _varlen_dk_last_head,
    "smallq_top_left": _smallq_top_left,
    "split_counts_floor": _split_counts_floor,
    "e4m3_bias_8": _e4m3_bias_8,
    "fp8_no_v_descale": _fp8_no_v_descale,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = _mutant(MUTANTS[name])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
