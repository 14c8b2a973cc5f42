"""The allocation-free decode entry point, for callers that cannot allocate.

A plugin that a host runtime calls with only its input and output buffers,
or a serving path whose device memory is planned up front, cannot hand the
decode a workspace. jfa_decode_splitkv_noalloc keeps the split partials in a
fixed scratch array inside the library instead. This test calls it through
the C ABI twice in a row, on different inputs, and checks each result against
the ordinary jfa_decode_splitkv (with its own workspace) within the parity
tolerances; it also checks that a request larger than the scratch is refused.
The file is collected last so a failure here cannot hide other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import _abi, inputs
from tests.parity import check_lse, check_o, np64

pytestmark = pytest.mark.gpu


def _args(q, kc, vc, pt, sl, splits, scale, o, lse):
    num_pages, P, Hkv, d = kc.shape
    return _abi.DecodeArgs(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pt.data_ptr(), sl.data_ptr(),
                           q.shape[0], q.shape[1], Hkv, d, P, num_pages, pt.shape[1], splits, scale,
                           o.data_ptr(), lse.data_ptr(), None, None)


def _case(seed, lens, page_size, splits, q_heads=32, kv_heads=8):
    d = inputs.decode_inputs(q_heads=q_heads, kv_heads=kv_heads, page_size=page_size, seed=seed, seqlens=lens)
    t = {k: d[k].cuda() for k in ("q", "k_cache", "v_cache", "page_table", "seqlens_k")}
    return d, t, splits


def test_noalloc_matches_workspace_entry_point_twice():
    lib = jfa.library()
    stream = torch.cuda.current_stream()
    cases = [_case(21, [1, 700, 0, 4097, 33], 16, 8), _case(22, [2049, 5, 128], 1, 3, q_heads=16, kv_heads=4)]
    for i, (d, t, S) in enumerate(cases):
        o_ref, lse_ref = jfa.jfa_decode_splitkv(t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["seqlens_k"],
                                                S, d["scale"], check=True)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        a = _args(t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["seqlens_k"], S, d["scale"], o, lse)
        st = lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream))
        assert st == _abi.JFA_OK, f"call {i}: status {st}"
        torch.cuda.synchronize()
        check_o(np64(o), np64(o_ref), f"noalloc O (call {i})")
        check_lse(np64(lse), np64(lse_ref), f"noalloc LSE (call {i})")


def test_noalloc_refuses_oversized_request():
    """num_splits * batch * q_heads above 32768 partial rows is refused up front."""
    lib = jfa.library()
    a = _abi.DecodeArgs(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 64, 32, 8, 128, 16, 100, 10, 32, 0.1,
                        0x10000, 0x10000, None, None)   # 32 * 64 * 32 = 65536 rows
    assert lib.jfa_decode_splitkv_noalloc(ctypes.byref(a), None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL
