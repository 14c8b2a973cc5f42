"""Per-role event trace of the persistent kernels: buffer, decoding, summary.

Only a library built with JFA_TRACE records (``build.build(variant="trace")``,
loaded when JFA_LIBRARY_VARIANT=trace is set before the first call); the
default library returns JFA_ERR_UNSUPPORTED from jfa_trace_enable. The record
layout and the event codes are those of csrc/trace.cuh: per CTA 16 warp
slots of ``records_per_warp`` records of 32 bytes (clock64, globaltimer,
event = kernel << 16 | code, argument, SM id, 0).

Times in the summary are SM cycles (clock64), compared only between warps of
the same CTA.
"""
from __future__ import annotations

import numpy as np

WARP_SLOTS = 16
RECORD_BYTES = 32

KERNELS = {1: "fwd_stream", 2: "bwd"}
EVENTS = {
    1: {1: "q_load", 2: "kv_load", 3: "s_issue", 4: "pv_issue", 5: "soft_begin", 6: "soft_end",
        7: "epi_begin", 8: "epi_end", 9: "soft_loaded", 10: "soft_pub", 11: "soft_exp", 12: "soft_max"},
    2: {1: "kv_load", 2: "q_load", 3: "item", 4: "s_issue", 5: "dp_issue", 6: "dv_issue", 7: "dqdk_issue",
        8: "p_begin", 9: "p_end", 10: "ds_begin", 11: "ds_end", 12: "dq_begin", 13: "dq_end",
        14: "acc_begin", 15: "acc_end"},
}
# warp index -> role, per kernel
ROLES = {
    1: {**{w: "softmax" for w in range(8)}, **{w: "epilogue" for w in range(8, 12)}, 12: "producer", 13: "mma"},
    2: {**{w: "softmax" for w in range(8)}, 8: "producer", 9: "mma", **{w: "epilogue" for w in range(10, 14)}},
}

RECORD_DTYPE = np.dtype([("clock", "<u8"), ("gtime", "<u8"), ("event", "<u4"), ("arg", "<u4"), ("smid", "<u4"),
                         ("zero", "<u4")])


def buffer_bytes(sms: int, records_per_warp: int) -> int:
    return sms * WARP_SLOTS * records_per_warp * RECORD_BYTES


def decode(raw: np.ndarray, records_per_warp: int) -> np.ndarray:
    """Records of a trace buffer (bytes) as a structured array with the fields
    cta, warp, seq (order within the warp), clock, gtime, kernel, code, arg, smid;
    empty records (clock and event 0) are dropped."""
    rec = np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=RECORD_DTYPE)
    n = rec.size
    slot = np.arange(n) // records_per_warp
    keep = (rec["event"] != 0) | (rec["clock"] != 0)
    out = np.zeros(int(keep.sum()), dtype=[("cta", "<i4"), ("warp", "<i4"), ("seq", "<i4"), ("clock", "<i8"),
                                           ("gtime", "<u8"), ("kernel", "<i4"), ("code", "<i4"), ("arg", "<i8"),
                                           ("smid", "<i4")])
    out["cta"] = (slot // WARP_SLOTS)[keep]
    out["warp"] = (slot % WARP_SLOTS)[keep]
    out["seq"] = (np.arange(n) % records_per_warp)[keep]
    out["clock"] = rec["clock"][keep].astype(np.int64)
    out["gtime"] = rec["gtime"][keep]
    out["kernel"] = (rec["event"][keep] >> 16).astype(np.int32)
    out["code"] = (rec["event"][keep] & 0xFFFF).astype(np.int32)
    out["arg"] = rec["arg"][keep]
    out["smid"] = rec["smid"][keep]
    return out


def counts(recs: np.ndarray) -> dict:
    """Number of records of every (kernel, event name)."""
    out = {}
    for kern, code in zip(recs["kernel"], recs["code"]):
        name = f"{KERNELS.get(int(kern), kern)}.{EVENTS.get(int(kern), {}).get(int(code), code)}"
        out[name] = out.get(name, 0) + 1
    return out


def _groups(recs):
    """{(cta, warp): that warp's records in program order}."""
    if recs.size == 0:
        return {}
    r = recs[np.lexsort((recs["seq"], recs["warp"], recs["cta"]))]
    key = r["cta"].astype(np.int64) * WARP_SLOTS + r["warp"]
    cut = np.flatnonzero(np.diff(key)) + 1
    return {(int(g["cta"][0]), int(g["warp"][0])): g for g in np.split(r, cut)}


def _code(g, code):
    sel = g[g["code"] == code]
    return sel["arg"], sel["clock"]


def _stats(values) -> dict:
    v = np.asarray(values, dtype=np.float64)
    if v.size == 0:
        return {"n": 0}
    return {"n": int(v.size), "median": float(np.median(v)), "mean": float(v.mean()), "p90": float(np.percentile(v, 90))}


def _paired(g, begin, end):
    """Durations end - begin of one warp's events, matched by argument."""
    a_b, c_b = _code(g, begin)
    a_e, c_e = _code(g, end)
    ends = dict(zip(a_e.tolist(), c_e.tolist()))
    return [ends[a] - c for a, c in zip(a_b.tolist(), c_b.tolist()) if a in ends]


def _paired_next(g, end, begin):
    """Gaps from an event `end` of step x to the event `begin` of step x + 1 of one warp."""
    a_e, c_e = _code(g, end)
    a_b, c_b = _code(g, begin)
    starts = dict(zip(a_b.tolist(), c_b.tolist()))
    return [starts[a + 1] - c for a, c in zip(a_e.tolist(), c_e.tolist()) if a + 1 in starts]


def summary_bwd(recs: np.ndarray) -> dict:
    """Per-role cycle statistics of the backward kernel over all CTAs:
    step: cycles between consecutive dQ/dK issues of the MMA warp within an item;
    item_gap: from the last dQ/dK issue of an item to the next item's first S^T issue
    (0 when that S^T was issued right after the last dQ);
    k_wait: from the last dQ/dK issue of an item to the MMA warp's start of the next item
    (its K has arrived);
    p_pass, ds_pass: softmax warps' P^T and dS passes; p_to_ds: from P^T stored to
    the start of the dS pass (waiting for dP^T or the dS buffer);
    dq_drain, acc_drain: epilogue's dQ and dK / dV drains."""
    step, gap, kwait, pp, dsp, p2d, dqd, accd = [], [], [], [], [], [], [], []
    for (cta, warp), g in _groups(recs[recs["kernel"] == 2]).items():
        if warp == 9:  # the MMA warp in program order: item (K arrived), S^T, dP^T, dV, dQ/dK issues
            item, last_item, last_dqdk, last_x = -1, -1, None, None
            s_at, bounds = {}, []
            for code, clk, arg in zip(g["code"].tolist(), g["clock"].tolist(), g["arg"].tolist()):
                if code == 3:
                    item = arg
                    if last_dqdk is not None:
                        kwait.append(clk - last_dqdk)
                        bounds.append((last_dqdk, last_x + 1))
                elif code == 4:
                    s_at.setdefault(arg, clk)
                elif code == 7:
                    if last_dqdk is not None and last_item == item:
                        step.append(clk - last_dqdk)
                    last_dqdk, last_item, last_x = clk, item, arg
            # the next item's first S^T may be recorded before its item event (issued early)
            gap += [s_at[x1] - c for c, x1 in bounds if x1 in s_at]
        elif warp < 8:
            pp += _paired(g, 8, 9)
            dsp += _paired(g, 10, 11)
            p2d += _paired(g, 9, 10)
        elif 10 <= warp < 14:
            dqd += _paired(g, 12, 13)
            accd += _paired(g, 14, 15)
    return {"step": _stats(step), "item_gap": _stats(gap), "k_wait": _stats(kwait), "p_pass": _stats(pp),
            "ds_pass": _stats(dsp), "p_to_ds": _stats(p2d), "dq_drain": _stats(dqd), "acc_drain": _stats(accd)}


def summary_fwd(recs: np.ndarray) -> dict:
    """Per-role cycle statistics of the forward-stream kernel over all CTAs:
    step: cycles between consecutive P V issues of the MMA warp;
    soft: softmax warps from S complete to P stored; s_to_soft: from the S
    issue to the start of that step's softmax (S in flight or queued);
    epi: epilogue from O complete to O and LSE written;
    soft_load / soft_max_pub / soft_exp / soft_other_max / soft_tail: the softmax step's phases
    (S read into registers; this half's maximum folded and published; the exponentials; waiting
    for and reading the other half's maximum; the rest up to P stored), soft_idle: from P stored
    to the next step's S complete."""
    step, soft, s2s, epi = [], [], [], []
    phases = {k: [] for k in ("load", "max_pub", "exp", "other_max", "tail", "idle")}
    groups = _groups(recs[recs["kernel"] == 1])
    s_issue = {}
    for (cta, warp), g in groups.items():
        if warp == 13:
            _, c_pv = _code(g, 4)
            step += np.diff(c_pv).tolist()
            a_s, c_s = _code(g, 3)
            s_issue[cta] = dict(zip(a_s.tolist(), c_s.tolist()))
    for (cta, warp), g in groups.items():
        if warp < 8:
            soft += _paired(g, 5, 6)
            phases["load"] += _paired(g, 5, 9)
            phases["max_pub"] += _paired(g, 9, 10)
            phases["idle"] += _paired_next(g, 6, 5)
            a_e, c_e = _code(g, 11)
            a_m, c_m = _code(g, 12)
            a_p, c_p = _code(g, 10)
            a_z, c_z = _code(g, 6)
            e_at, m_at, p_at, z_at = (dict(zip(a.tolist(), c.tolist())) for a, c in
                                      ((a_e, c_e), (a_m, c_m), (a_p, c_p), (a_z, c_z)))
            for x_, ce in e_at.items():
                if x_ in m_at and x_ in p_at and x_ in z_at:
                    if ce <= m_at[x_]:  # exponentials first (speculative), then the other maximum
                        phases["exp"].append(ce - p_at[x_])
                        phases["other_max"].append(m_at[x_] - ce)
                        phases["tail"].append(z_at[x_] - m_at[x_])
                    else:               # first step of an item: the other maximum first
                        phases["other_max"].append(m_at[x_] - p_at[x_])
                        phases["exp"].append(ce - m_at[x_])
                        phases["tail"].append(z_at[x_] - ce)
            s_at = s_issue.get(cta, {})
            a_b, c_b = _code(g, 5)
            s2s += [c - s_at[a] for a, c in zip(a_b.tolist(), c_b.tolist()) if a in s_at]
        elif 8 <= warp < 12:
            epi += _paired(g, 7, 8)
    out = {"step": _stats(step), "soft": _stats(soft), "s_to_soft": _stats(s2s), "epi": _stats(epi)}
    out.update({f"soft_{k}": _stats(v) for k, v in phases.items()})
    return out
