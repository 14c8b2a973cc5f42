"""The allocation-free decode entry point, for callers that cannot allocate.

A plugin that a host runtime calls with only its input and output buffers,
or a serving path whose device memory is planned up front, cannot hand the
decode a workspace. jfa_decode_splitkv_noalloc keeps the split partials in a
fixed scratch array inside the library instead. These tests call it through
the C ABI:
  - twice in a row, on different inputs, each result bit for bit equal to the
    ordinary jfa_decode_splitkv (same kernels, same partial layout, its own
    workspace) and within the parity tolerances of the fp64 oracle;
  - at exactly the scratch limit (num_splits * batch * q_heads = 32768 rows);
  - a few more times with the device's free memory read before and after
    (nothing may be allocated);
  - with a page-table entry out of range, whose device-detected status is read
    back through jfa_decode_noalloc_status;
and check that a request larger than the scratch is refused. The file is
collected last, so a failure here cannot hide other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.attention as orc
import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import _abi, inputs
from tests.parity import check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _args(t, splits, scale, o, lse):
    num_pages, P, Hkv, d = t["k_cache"].shape
    q = t["q"]
    return _abi.DecodeArgs(q.data_ptr(), t["k_cache"].data_ptr(), t["v_cache"].data_ptr(), t["page_table"].data_ptr(),
                           t["seqlens_k"].data_ptr(), q.shape[0], q.shape[1], Hkv, d, P, num_pages,
                           t["page_table"].shape[1], splits, scale, o.data_ptr(), lse.data_ptr(), None, None)


def _case(seed, lens, page_size, splits, q_heads=32, kv_heads=8):
    d = inputs.decode_inputs(q_heads=q_heads, kv_heads=kv_heads, page_size=page_size, seed=seed, seqlens=lens)
    t = {k: d[k].cuda() for k in ("q", "k_cache", "v_cache", "page_table", "seqlens_k")}
    return d, t, splits


def _noalloc(t, S, scale, like_o, like_lse):
    """One call of the allocation-free entry point on the current stream."""
    lib = jfa.library()
    o = torch.full_like(like_o, float("nan"))
    lse = torch.full_like(like_lse, float("nan"))
    a = _args(t, S, scale, o, lse)
    st = lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


def _oracle(d):
    return orc.decode_forward(np64(d["q"]), np64(d["k_cache"]), np64(d["v_cache"]), d["page_table"].numpy(),
                              d["seqlens_k"].numpy(), d["page_size"], d["scale"])


def _check_against_both(d, t, S, what):
    o_ref, lse_ref = jfa.jfa_decode_splitkv(t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["seqlens_k"],
                                            S, d["scale"], check=True)
    st, o, lse = _noalloc(t, S, d["scale"], o_ref, lse_ref)
    assert st == _abi.JFA_OK, f"{what}: status {st}"
    torch.cuda.synchronize()
    # the same kernels on the same inputs: bit for bit the workspace entry point's result
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"{what}: O differs from jfa_decode_splitkv"
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), f"{what}: LSE differs"
    O_or, L_or = _oracle(d)
    check_o(np64(o), O_or, f"{what}: O against the oracle")
    check_lse(np64(lse), L_or, f"{what}: LSE against the oracle")
    st, det = _status()
    assert st == _abi.JFA_OK, (st, det)


def _status():
    det = ctypes.c_int32(-1)
    st = jfa.library().jfa_decode_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                                 ctypes.byref(det))
    return st, det.value


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [_case(21, [1, 700, 0, 4097, 33], 16, 8), _case(22, [2049, 5, 128], 1, 3, q_heads=16, kv_heads=4)]
    for i, (d, t, S) in enumerate(cases):
        _check_against_both(d, t, S, f"call {i}")


def test_noalloc_at_the_scratch_limit():
    """num_splits * batch * q_heads = 32 * 32 * 32 = 32768 partial rows, the
    largest request the scratch takes."""
    g = np.random.default_rng(23)
    lens = g.integers(0, 300, size=32).tolist()
    d, t, S = _case(23, lens, 16, 32)
    assert S * t["q"].shape[0] * t["q"].shape[1] == 32768
    _check_against_both(d, t, S, "32768 rows")


def test_noalloc_allocates_nothing():
    d, t, S = _case(24, [513, 2, 1200], 16, 16)
    o_ref, lse_ref = jfa.jfa_decode_splitkv(t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["seqlens_k"],
                                            S, d["scale"], check=True)
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    a = _args(t, S, d["scale"], o, lse)
    lib = jfa.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), stream) == _abi.JFA_OK  # first call: set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(4):
        assert lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), stream) == _abi.JFA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))


def test_noalloc_reports_a_bad_page_table():
    """A page index past num_pages: the kernel substitutes page 0 (every access
    stays in bounds) and records JFA_ERR_BAD_INPUT in the scratch's status word."""
    d = inputs.decode_inputs(q_heads=8, kv_heads=2, page_size=4, seed=5, seqlens=[9, 4])
    d["page_table"][0, 1] = d["num_pages"] + 5
    t = {k: d[k].cuda() for k in ("q", "k_cache", "v_cache", "page_table", "seqlens_k")}
    like_o = torch.empty_like(t["q"])
    like_lse = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    st, _, _ = _noalloc(t, 2, d["scale"], like_o, like_lse)
    assert st == _abi.JFA_OK
    st, det = _status()
    assert st == _abi.JFA_ERR_BAD_INPUT, (st, det)
    # the next good call clears the status again
    d2, t2, S = _case(25, [40, 7], 16, 2, q_heads=8, kv_heads=2)
    _check_against_both(d2, t2, S, "after the bad call")


def test_noalloc_refuses_oversized_request():
    """num_splits * batch * q_heads above 32768 partial rows is refused up front."""
    lib = jfa.library()
    a = _abi.DecodeArgs(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 64, 32, 8, 128, 16, 100, 10, 32, 0.1,
                        0x10000, 0x10000, None, None)   # 32 * 64 * 32 = 65536 rows
    assert lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL
