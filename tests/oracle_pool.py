"""Full-size parity checks fanned out over the host cores.

The fp64 oracle (oracle/attention.py) is called unchanged, once per chunk of
whole sequences, in a pool of spawned worker processes (spawned, not forked:
the parent holds a CUDA context). Each worker gets its chunk's bf16 inputs
and the GPU's outputs as raw 16-bit words, runs the oracle on the chunk and
returns only error statistics, so no full-size fp64 array is ever built or
sent back. The parent applies the stated tolerances:
  O      |gpu - oracle| <= 1e-2 + 2^-7 |oracle|   elementwise
  LSE    max|gpu - oracle| <= 1e-3
  dQ, dK, dV   max|gpu - oracle| <= 2e-2 * max|oracle| over the whole tensor
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

from tests.parity import TOL_GRAD_REL, TOL_LSE, TOL_O, TOL_O_REL


def _workers(mem_per_worker_gb: float = 2.0) -> int:
    n = os.cpu_count() or 4
    try:
        mem_gb = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES") / 2 ** 30
        n = min(n, max(1, int(mem_gb * 0.5 / mem_per_worker_gb)))
    except (ValueError, OSError, AttributeError):
        pass
    return max(1, n)


def pool(mem_per_worker_gb: float = 2.0) -> cf.ProcessPoolExecutor:
    """A spawned pool whose workers run single-threaded BLAS (one core each).

    The thread-count variables are set in this process's environment (its own
    BLAS is already loaded, so they only reach new processes) and every worker
    is started at once, so none is spawned later without them."""
    import time
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    n = _workers(mem_per_worker_gb)
    ex = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
    list(ex.map(time.sleep, [0.5] * n))  # n tasks in flight at once: one worker each
    return ex


def raw16(t) -> np.ndarray:
    """The 16-bit words of a bf16 torch tensor (no conversion)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy()


def bf16_words_to_f64(w: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly."""
    return (w.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- worker side

def _o_stats(gpu, ref):
    """(max over elements of |diff| - bound, max |diff|, elements above the plain 1e-2, elements)."""
    if ref.size == 0:
        return -np.inf, 0.0, 0, 0
    diff = np.abs(gpu - ref)
    diff = np.where(np.isnan(diff), np.inf, diff)
    return (float(np.max(diff - (TOL_O + TOL_O_REL * np.abs(ref)))), float(diff.max()),
            int(np.count_nonzero(diff > TOL_O)), int(diff.size))


def _max_err(a, b):
    if a.size == 0:
        return 0.0
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    return float(np.where(np.isnan(d), np.inf, d).max())


def _grad_stats(gpu, ref):
    return (_max_err(gpu, ref), float(np.abs(ref).max()) if ref.size else 0.0)


def self_chunk(job):
    """One chunk of jagged self-attention: oracle forward + backward of the
    chunk's sequences, compared with the GPU's outputs."""
    import oracle.attention as orc
    (q, k, v, do, o, lse, dq, dk, dv, off, scale, causal) = job
    q, k, v, do = (bf16_words_to_f64(x) for x in (q, k, v, do))
    O, L = orc.attention_forward(q, k, v, off, scale, causal)
    dQ, dK, dV, _ = orc.attention_backward(q, k, v, do, off, scale, causal)
    return {"o": _o_stats(bf16_words_to_f64(o), O), "lse": _max_err(lse.astype(np.float64), L),
            "dq": _grad_stats(bf16_words_to_f64(dq), dQ), "dk": _grad_stats(bf16_words_to_f64(dk), dK),
            "dv": _grad_stats(bf16_words_to_f64(dv), dV), "rows": int(off[-1])}


def bcast_chunk(job):
    """A chunk of broadcast-Q sequences: O, LSE, dK, dV compared; the chunk's
    part of the dQ sum returned for the parent to add up."""
    import oracle.attention as orc
    (q, k, v, do, o, lse, dk, dv, off, scale) = job
    q, k, v, do = (bf16_words_to_f64(x) for x in (q, k, v, do))
    O, L = orc.broadcast_forward(q, k, v, off, scale)
    dQ, dK, dV = orc.broadcast_backward(q, k, v, do, off, scale)
    return {"o": _o_stats(bf16_words_to_f64(o), O), "lse": _max_err(lse.astype(np.float64), L),
            "dk": _grad_stats(bf16_words_to_f64(dk), dK), "dv": _grad_stats(bf16_words_to_f64(dv), dV),
            "dq_part": dQ}


# ---------------------------------------------------------------- parent side

def _chunks(offsets, max_rows):
    """Consecutive runs of whole sequences with about max_rows rows each."""
    off = [int(x) for x in offsets]
    out, b0 = [], 0
    for b in range(len(off) - 1):
        if off[b + 1] - off[b0] >= max_rows or b == len(off) - 2:
            out.append((b0, b + 1))
            b0 = b + 1
    return [c for c in out if c[1] > c[0]]


def _assert_stats(stats, what, grads):
    from tests.parity import report_plain_o
    viol = max(s["o"][0] for s in stats)
    assert viol <= 0.0, f"{what}: O exceeds 1e-2 + 2^-7|O| by {viol:.3e} (max|diff| {max(s['o'][1] for s in stats):.3e})"
    report_plain_o(f"{what} O", sum(s["o"][2] for s in stats), sum(s["o"][3] for s in stats),
                   max(s["o"][1] for s in stats))
    e = max(s["lse"] for s in stats)
    assert e <= TOL_LSE, f"{what}: LSE max|diff| {e:.3e} > {TOL_LSE}"
    for g in grads:
        err = max(s[g][0] for s in stats)
        ref = max(s[g][1] for s in stats)
        assert err <= TOL_GRAD_REL * ref or (ref == 0.0 and err == 0.0), \
            f"{what}: {g} max|diff| {err:.3e} > {TOL_GRAD_REL} * max|ref| ({ref:.3e})"


def check_self_full(ex, d, gpu, causal, what, max_rows=8192):
    """Every sequence of a jagged self-attention batch: d holds the CPU bf16
    inputs and offsets, gpu = (o, lse, dq, dk, dv) on the device."""
    o, lse, dq, dk, dv = gpu
    words = {x: raw16(d[x]) for x in ("q", "k", "v", "do")}
    out = {"o": raw16(o), "dq": raw16(dq), "dk": raw16(dk), "dv": raw16(dv)}
    lse_h = lse.detach().float().cpu().numpy()
    off = d["offsets"].numpy()
    jobs = []
    for b0, b1 in _chunks(off, max_rows):
        s0, s1 = int(off[b0]), int(off[b1])
        sub_off = off[b0:b1 + 1] - s0
        jobs.append(tuple(words[x][s0:s1] for x in ("q", "k", "v", "do")) +
                    (out["o"][s0:s1], lse_h[:, s0:s1], out["dq"][s0:s1], out["dk"][s0:s1], out["dv"][s0:s1],
                     sub_off, d["scale"], causal))
    stats = list(ex.map(self_chunk, jobs))
    assert sum(s["rows"] for s in stats) == int(off[-1])
    _assert_stats(stats, what, ("dq", "dk", "dv"))


def check_self_pairs(ex, d, gpu, pairs, causal, what):
    """Whole (sequence, head) pairs of a jagged self-attention batch, one job each."""
    o, lse, dq, dk, dv = gpu
    lse_h = lse.detach().float().cpu().numpy()
    off = d["offsets"].numpy()
    jobs = []
    for b, h in pairs:
        s0, s1 = int(off[b]), int(off[b + 1])
        sl = lambda t: raw16(t[s0:s1, h:h + 1])  # noqa: E731
        jobs.append((sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["do"]), sl(o), lse_h[h:h + 1, s0:s1], sl(dq), sl(dk),
                     sl(dv), np.array([0, s1 - s0]), d["scale"], causal))
    stats = list(ex.map(self_chunk, jobs))
    _assert_stats(stats, what, ("dq", "dk", "dv"))


def check_bcast_full(ex, d, gpu, what, seqs_per_chunk=16):
    """Every sequence of a broadcast-Q batch, and the dQ summed over all of them."""
    o, lse, dq, dk, dv = gpu
    q = raw16(d["q"])
    kw, vw, dow = raw16(d["k"]), raw16(d["v"]), raw16(d["do"])
    ow, dkw, dvw = raw16(o), raw16(dk), raw16(dv)
    lse_h = lse.detach().float().cpu().numpy()
    off = d["kv_offsets"].numpy()
    B = len(off) - 1
    jobs = []
    for b0 in range(0, B, seqs_per_chunk):
        b1 = min(B, b0 + seqs_per_chunk)
        s0, s1 = int(off[b0]), int(off[b1])
        jobs.append((q, kw[s0:s1], vw[s0:s1], dow[b0:b1], ow[b0:b1], lse_h[b0:b1], dkw[s0:s1], dvw[s0:s1],
                     off[b0:b1 + 1] - s0, d["scale"]))
    stats = list(ex.map(bcast_chunk, jobs))
    _assert_stats(stats, what, ("dk", "dv"))
    dQ = sum(s["dq_part"] for s in stats)
    dq64 = bf16_words_to_f64(raw16(dq))
    e, ref = _max_err(dq64, dQ), float(np.abs(dQ).max())
    assert e <= TOL_GRAD_REL * ref, f"{what}: dQ (sum over {B}) max|diff| {e:.3e} > {TOL_GRAD_REL} * {ref:.3e}"
