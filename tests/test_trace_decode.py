"""The trace decoder and its summaries on a hand-built record buffer (CPU): record layout,
the event names, and the per-role durations of a known event sequence."""
import numpy as np

from varlen_flashattention_gb300 import trace

CAP = 16


def _buffer(events):
    """events: (cta, warp, clock, kernel, code, arg) in program order per warp."""
    ctas = 1 + max(e[0] for e in events)
    rec = np.zeros(ctas * trace.WARP_SLOTS * CAP, dtype=trace.RECORD_DTYPE)
    n = {}
    for cta, warp, clk, kern, code, arg in events:
        slot = cta * trace.WARP_SLOTS + warp
        i = n.get(slot, 0)
        n[slot] = i + 1
        r = rec[slot * CAP + i]
        r["clock"], r["gtime"], r["event"], r["arg"], r["smid"] = clk, 1000 + clk, kern << 16 | code, arg, 7
        rec[slot * CAP + i] = r
    return rec.view(np.uint8)


# one backward CTA: item 0 with steps 0 and 1, item 1 with step 2
BWD = [
    (0, 9, 100, 2, 3, 0), (0, 9, 110, 2, 4, 0), (0, 9, 120, 2, 5, 0), (0, 9, 300, 2, 6, 0), (0, 9, 500, 2, 7, 0),
    (0, 9, 500, 2, 4, 1), (0, 9, 520, 2, 5, 1), (0, 9, 700, 2, 6, 1), (0, 9, 900, 2, 7, 1),
    (0, 9, 1200, 2, 3, 1), (0, 9, 1210, 2, 4, 2), (0, 9, 1220, 2, 5, 2), (0, 9, 1400, 2, 6, 2), (0, 9, 1500, 2, 7, 2),
    (0, 0, 200, 2, 8, 0), (0, 0, 280, 2, 9, 0), (0, 0, 350, 2, 10, 0), (0, 0, 450, 2, 11, 0),
    (0, 10, 600, 2, 12, 0), (0, 10, 660, 2, 13, 0), (0, 10, 1000, 2, 14, 0), (0, 10, 1150, 2, 15, 0),
]


def test_decode_layout_and_names():
    recs = trace.decode(_buffer(BWD), CAP)
    assert recs.size == len(BWD)
    m = recs[(recs["warp"] == 9)]
    m = m[np.argsort(m["seq"])]
    assert m["clock"].tolist() == [e[2] for e in BWD if e[1] == 9]
    assert set(recs["smid"].tolist()) == {7} and set(recs["cta"].tolist()) == {0}
    assert np.all(recs["gtime"] == recs["clock"] + 1000)
    c = trace.counts(recs)
    assert c["bwd.item"] == 2 and c["bwd.s_issue"] == 3 and c["bwd.dqdk_issue"] == 3 and c["bwd.p_begin"] == 1


def test_backward_summary_of_a_known_sequence():
    s = trace.summary_bwd(trace.decode(_buffer(BWD), CAP))
    assert s["step"]["n"] == 1 and s["step"]["median"] == 400      # dQ/dK issues of steps 0 and 1 (item 0)
    assert s["k_wait"]["median"] == 300                              # last dQ/dK of item 0 -> K of item 1
    assert s["item_gap"]["median"] == 310                            # -> first S^T of item 1
    assert s["p_pass"]["median"] == 80 and s["ds_pass"]["median"] == 100 and s["p_to_ds"]["median"] == 70
    assert s["dq_drain"]["median"] == 60 and s["acc_drain"]["median"] == 150


def test_forward_summary_of_a_known_sequence():
    ev = [(0, 13, 100, 1, 3, 0), (0, 13, 150, 1, 3, 1), (0, 13, 400, 1, 4, 0), (0, 13, 450, 1, 3, 2),
          (0, 13, 900, 1, 4, 1), (0, 4, 200, 1, 5, 0), (0, 4, 380, 1, 6, 0), (0, 4, 600, 1, 5, 1),
          (0, 4, 850, 1, 6, 1), (0, 8, 950, 1, 7, 0), (0, 8, 1100, 1, 8, 0)]
    s = trace.summary_fwd(trace.decode(_buffer(ev), CAP))
    assert s["step"]["median"] == 500
    assert sorted([180, 250]) == [180, 250] and s["soft"]["n"] == 2 and s["soft"]["mean"] == 215
    assert s["s_to_soft"]["n"] == 2 and s["s_to_soft"]["mean"] == (100 + 450) / 2
    assert s["epi"]["median"] == 150
