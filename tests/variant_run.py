"""Checks of the debugging builds, run in a child process (python -m tests.variant_run trace|debug)
with JFA_LIBRARY_VARIANT set, so that the package loads libjfa_trace.so / libjfa_debug.so.

trace: forward and backward of a jagged batch with tracing on; every role records one event
       per step or item (counts derived from the lengths), each warp's cycle stamps never
       decrease, and the results still match the fp64 oracle.
debug: the parity cases of the persistent kernels (self-attention at head_dim 64, 128 and 192,
       causal and not; varlen GQA; broadcast-Q; the FP8 forward) with every tile load checked;
       the status is OK and the results match the oracle.
Exits non-zero on the first failure.
"""
from __future__ import annotations

import math
import os
import sys

import numpy as np
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import inputs, trace
from tests.parity import check_grad, check_lse, check_o, fp8_error_bound, np64

LENGTHS = [300, 128, 1, 513, 77, 256, 0, 129]


def _case(lengths, heads, head_dim, seed):
    g = torch.Generator().manual_seed(seed)
    return inputs.jagged_from_lengths(torch.tensor(lengths, dtype=torch.int32), heads, head_dim, g)


def _self(d, causal, head_chunk=0, between=None):
    q, k, v, off, do = (d[x].cuda() for x in ("q", "k", "v", "offsets", "do"))
    o, lse = jfa.jfa_fwd(q, k, v, off, d["max_seqlen"], d["scale"], causal, check=True)
    if between is not None:
        between()
    dq, dk, dv = jfa.jfa_bwd(q, k, v, o, do, lse, off, d["max_seqlen"], d["scale"], causal, head_chunk, check=True)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def _check_self(d, causal, res, tag):
    o, lse, dq, dk, dv = res
    q, k, v, do = (np64(d[x]) for x in ("q", "k", "v", "do"))
    off = d["offsets"].numpy()
    O, L = orc.attention_forward(q, k, v, off, d["scale"], causal)
    check_o(np64(o), O, f"O {tag}")
    check_lse(np64(lse), L, f"LSE {tag}")
    dQ, dK, dV, _ = orc.attention_backward(q, k, v, do, off, d["scale"], causal)
    check_grad(np64(dq), dQ, f"dQ {tag}")
    check_grad(np64(dk), dK, f"dK {tag}")
    check_grad(np64(dv), dV, f"dV {tag}")


def run_trace():
    assert jfa.jfa_trace_compiled() == 1, "the trace build is not the one loaded"
    heads, cap = 2, 512
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(trace.buffer_bytes(sms, cap), dtype=torch.uint8, device="cuda")
    d = _case(LENGTHS, heads, 128, seed=5)
    nt = [math.ceil(L / 128) for L in LENGTHS]
    steps = heads * sum(t * t for t in nt)  # non-causal: every (query tile, key tile) pair of a sequence
    items = heads * sum(nt)                 # forward: query tiles; backward: key tiles
    recs = {}

    def grab(tag):
        torch.cuda.synchronize()
        recs[tag] = trace.decode(buf.cpu().numpy(), cap)
        buf.zero_()

    jfa.jfa_trace_enable(buf, cap)
    res = _self(d, False, between=lambda: grab("fwd"))
    grab("bwd")
    jfa.jfa_trace_enable(None)
    _check_self(d, False, res, "trace build")

    f = trace.counts(recs["fwd"])
    want_f = {"fwd_stream.q_load": items, "fwd_stream.kv_load": 2 * steps, "fwd_stream.s_issue": steps,
              "fwd_stream.pv_issue": steps, "fwd_stream.soft_begin": 8 * steps, "fwd_stream.soft_end": 8 * steps,
              "fwd_stream.epi_begin": 4 * items, "fwd_stream.epi_end": 4 * items,
              "fwd_stream.soft_loaded": 8 * steps, "fwd_stream.soft_pub": 8 * steps, "fwd_stream.soft_exp": 8 * steps,
              "fwd_stream.soft_max": 8 * steps}
    assert f == want_f, f"forward event counts {f} != {want_f}"
    b = trace.counts(recs["bwd"])
    want_b = {"bwd.kv_load": items, "bwd.q_load": steps, "bwd.item": items, "bwd.s_issue": steps,
              "bwd.dp_issue": steps, "bwd.dv_issue": steps, "bwd.dqdk_issue": steps, "bwd.p_begin": 8 * steps,
              "bwd.p_end": 8 * steps, "bwd.ds_begin": 8 * steps, "bwd.ds_end": 8 * steps,
              "bwd.dq_begin": 4 * steps, "bwd.dq_end": 4 * steps, "bwd.acc_begin": 4 * items,
              "bwd.acc_end": 4 * items}
    assert b == want_b, f"backward event counts {b} != {want_b}"
    for tag, r in recs.items():
        for cta, warp in {(int(c), int(w)) for c, w in zip(r["cta"], r["warp"])}:
            m = r[(r["cta"] == cta) & (r["warp"] == warp)]
            m = m[np.argsort(m["seq"])]
            assert np.all(np.diff(m["clock"]) >= 0), f"{tag}: CTA {cta} warp {warp}: cycle stamps decrease"
            assert np.all(m["seq"] == np.arange(m.size)), f"{tag}: CTA {cta} warp {warp}: records not contiguous"
            assert np.unique(m["smid"]).size == 1, f"{tag}: CTA {cta} warp {warp}: more than one SM"
    sb, sf = trace.summary_bwd(recs["bwd"]), trace.summary_fwd(recs["fwd"])
    assert sb["step"]["n"] > 0 and sb["p_pass"]["median"] > 0 and sf["soft"]["median"] > 0
    # recording off: nothing is written
    _self(d, False)
    assert int(buf.count_nonzero()) == 0, "records written after jfa_trace_enable(None)"
    print("trace ok", {"bwd step median": sb["step"].get("median"), "fwd step median": sf["step"].get("median")})


def run_debug():
    assert jfa.jfa_trace_compiled() == 0
    for head_dim, causal, chunk in ((128, False, 0), (128, True, 0), (64, True, 0), (192, False, 0), (192, True, 64)):
        d = _case(LENGTHS, 2, head_dim, seed=head_dim + causal)
        _check_self(d, causal, _self(d, causal, chunk), f"debug build d={head_dim} causal={causal} chunk={chunk}")
    # varlen GQA, bottom-right causal
    g = torch.Generator().manual_seed(11)
    dv_ = inputs.varlen_from_lengths([200, 1, 0, 384], [300, 129, 5, 384], 4, 2, 128, g)
    q, k, v, do, qo, ko = (dv_[x].cuda() for x in ("q", "k", "v", "do", "q_offsets", "k_offsets"))
    o, lse = jfa.jfa_fwd_varlen(q, k, v, qo, ko, dv_["max_seqlen_q"], dv_["max_seqlen_k"], dv_["scale"], True,
                                check=True)
    dq, dk, dv = jfa.jfa_bwd_varlen(q, k, v, o, do, lse, qo, ko, dv_["max_seqlen_q"], dv_["max_seqlen_k"],
                                    dv_["scale"], True, check=True)
    args = [np64(dv_[x]) for x in ("q", "k", "v")]
    O, L = orc.varlen_forward(*args, dv_["q_offsets"].numpy(), dv_["k_offsets"].numpy(), dv_["scale"], True)
    check_o(np64(o), O, "O varlen debug build")
    check_lse(np64(lse), L, "LSE varlen debug build")
    dQ, dK, dV = orc.varlen_backward(*args, np64(dv_["do"]), dv_["q_offsets"].numpy(), dv_["k_offsets"].numpy(),
                                     dv_["scale"], True)
    check_grad(np64(dq), dQ, "dQ varlen debug build")
    check_grad(np64(dk), dK, "dK varlen debug build")
    check_grad(np64(dv), dV, "dV varlen debug build")
    # broadcast-Q
    bq = inputs.broadcast_inputs(batch=6, q_len=200, heads=2, head_dim=128, lk_lo=1, lk_hi=300, seed=3)
    q, k, v, do, ko = (bq[x].cuda() for x in ("q", "k", "v", "do", "kv_offsets"))
    o, lse = jfa.jfa_fwd_broadcast_q(q, k, v, ko, bq["max_seqlen_k"], bq["scale"], check=True)
    dq, dk, dv = jfa.jfa_bwd_broadcast_q(q, k, v, o, do, lse, ko, bq["max_seqlen_k"], bq["scale"], check=True)
    args = [np64(bq[x]) for x in ("q", "k", "v")]
    O, L = orc.broadcast_forward(*args, bq["kv_offsets"].numpy(), bq["scale"])
    check_o(np64(o), O, "O broadcast debug build")
    check_lse(np64(lse), L, "LSE broadcast debug build")
    dQ, dK, dV = orc.broadcast_backward(*args, np64(bq["do"]), bq["kv_offsets"].numpy(), bq["scale"])
    check_grad(np64(dq), dQ, "dQ broadcast debug build")
    check_grad(np64(dk), dK, "dK broadcast debug build")
    check_grad(np64(dv), dV, "dV broadcast debug build")
    # FP8 forward (its own kernel and V transpose pass), within the derived bound
    for causal in (False, True):
        d8 = inputs.fp8_from_lengths(LENGTHS, 2, seed=17)
        q, k, v, off = (d8[x].cuda() for x in ("q", "k", "v", "offsets"))
        o, lse = jfa.jfa_fwd_fp8(q, k, v, off, d8["max_seqlen"], d8["q_descale"], d8["k_descale"], d8["v_descale"],
                                 d8["scale"], causal, check=True)
        q8, k8, v8 = (d8[x].numpy() for x in ("q", "k", "v"))
        qd, kd, vd = d8["q_descale"], d8["k_descale"], d8["v_descale"]
        O, L = orc.attention_forward_fp8(q8, k8, v8, d8["offsets"].numpy(), d8["scale"], causal, qd, kd, vd)
        check_lse(np64(lse), L, f"LSE fp8 debug build causal={causal}")
        bound = fp8_error_bound(orc.e4m3_decode(q8) * qd, orc.e4m3_decode(k8) * kd, orc.e4m3_decode(v8) * vd,
                                d8["offsets"].numpy(), d8["scale"], causal, O)
        assert np.all(np.abs(np64(o) - O) <= bound), f"O fp8 debug build causal={causal} outside the bound"
    print("debug ok")


if __name__ == "__main__":
    mode = sys.argv[1]
    assert os.environ.get("JFA_LIBRARY_VARIANT") == mode, "run with JFA_LIBRARY_VARIANT set to the mode"
    {"trace": run_trace, "debug": run_debug}[mode]()
