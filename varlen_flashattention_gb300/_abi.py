"""ctypes mirror of include/jfa.h: structures, status codes and the loaded library.

Only argument marshalling lives here; every step of the computation runs in
the CUDA kernels of libjfa.so. If the library has not been built, loading it
raises (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjfa.so")
# A debugging build of the same sources to load instead ("trace" or "debug",
# made by build.build(variant=...)); read once, at the first load.
VARIANT_ENV = "JFA_LIBRARY_VARIANT"

c_void_p = ctypes.c_void_p
c_i32 = ctypes.c_int32
c_f32 = ctypes.c_float

JFA_OK = 0
JFA_ERR_INVALID_ARG = 1
JFA_ERR_UNSUPPORTED = 2
JFA_ERR_WORKSPACE_TOO_SMALL = 3
JFA_ERR_CUDA = 4
JFA_ERR_TIMEOUT = 5
JFA_ERR_BAD_INPUT = 6


class FwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("offsets", c_void_p),
                ("batch", c_i32), ("heads", c_i32), ("head_dim", c_i32), ("max_seqlen", c_i32),
                ("total", c_i32), ("scale", c_f32), ("causal", c_i32),
                ("o", c_void_p), ("lse", c_void_p), ("main_kernel_events", c_void_p)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("o", c_void_p), ("dout", c_void_p),
                ("lse", c_void_p), ("offsets", c_void_p),
                ("batch", c_i32), ("heads", c_i32), ("head_dim", c_i32), ("max_seqlen", c_i32),
                ("total", c_i32), ("scale", c_f32), ("causal", c_i32), ("head_chunk", c_i32),
                ("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p), ("main_kernel_events", c_void_p)]


class BcastFwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("kv_offsets", c_void_p),
                ("batch", c_i32), ("q_len", c_i32), ("heads", c_i32), ("head_dim", c_i32),
                ("max_seqlen_k", c_i32), ("total_k", c_i32), ("scale", c_f32),
                ("o", c_void_p), ("lse", c_void_p), ("main_kernel_events", c_void_p)]


class BcastBwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("o", c_void_p), ("dout", c_void_p),
                ("lse", c_void_p), ("kv_offsets", c_void_p),
                ("batch", c_i32), ("q_len", c_i32), ("heads", c_i32), ("head_dim", c_i32),
                ("max_seqlen_k", c_i32), ("total_k", c_i32), ("scale", c_f32),
                ("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p), ("main_kernel_events", c_void_p)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k_cache", c_void_p), ("v_cache", c_void_p), ("page_table", c_void_p),
                ("seqlens_k", c_void_p),
                ("batch", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
                ("page_size", c_i32), ("num_pages", c_i32), ("max_pages", c_i32), ("num_splits", c_i32),
                ("scale", c_f32),
                ("o", c_void_p), ("lse", c_void_p), ("split_bounds_out", c_void_p),
                ("main_kernel_events", c_void_p)]


class VarlenFwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("q_offsets", c_void_p), ("k_offsets", c_void_p),
                ("batch", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
                ("max_seqlen_q", c_i32), ("max_seqlen_k", c_i32), ("total_q", c_i32), ("total_k", c_i32),
                ("scale", c_f32), ("causal", c_i32),
                ("o", c_void_p), ("lse", c_void_p), ("main_kernel_events", c_void_p)]


class VarlenBwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("o", c_void_p), ("dout", c_void_p),
                ("lse", c_void_p), ("q_offsets", c_void_p), ("k_offsets", c_void_p),
                ("batch", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
                ("max_seqlen_q", c_i32), ("max_seqlen_k", c_i32), ("total_q", c_i32), ("total_k", c_i32),
                ("scale", c_f32), ("causal", c_i32), ("head_chunk", c_i32),
                ("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p), ("main_kernel_events", c_void_p)]


class DecodeSmallqArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k_cache", c_void_p), ("v_cache", c_void_p), ("page_table", c_void_p),
                ("seqlens_k", c_void_p),
                ("batch", c_i32), ("q_len", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
                ("page_size", c_i32), ("num_pages", c_i32), ("max_pages", c_i32), ("num_splits", c_i32),
                ("min_split_tokens", c_i32), ("scale", c_f32),
                ("o", c_void_p), ("lse", c_void_p), ("split_bounds_out", c_void_p), ("split_counts_out", c_void_p),
                ("main_kernel_events", c_void_p)]


class FwdFp8Args(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("offsets", c_void_p),
                ("batch", c_i32), ("heads", c_i32), ("head_dim", c_i32), ("max_seqlen", c_i32), ("total", c_i32),
                ("scale", c_f32), ("causal", c_i32), ("q_descale", c_f32), ("k_descale", c_f32),
                ("v_descale", c_f32), ("o", c_void_p), ("lse", c_void_p), ("main_kernel_events", c_void_p),
                ("vt", c_void_p)]


class Fp8QuantizeVArgs(ctypes.Structure):
    _fields_ = [("v", c_void_p), ("offsets", c_void_p), ("batch", c_i32), ("heads", c_i32), ("head_dim", c_i32),
                ("max_seqlen", c_i32), ("total", c_i32), ("v_descale", c_f32), ("vt", c_void_p)]


# (name, argtypes, restype) of every exported symbol declared in include/jfa.h
SIGNATURES = [
    ("jfa_fwd_workspace_size", [ctypes.POINTER(FwdArgs)], ctypes.c_size_t),
    ("jfa_bwd_workspace_size", [ctypes.POINTER(BwdArgs)], ctypes.c_size_t),
    ("jfa_bcast_fwd_workspace_size", [ctypes.POINTER(BcastFwdArgs)], ctypes.c_size_t),
    ("jfa_bcast_bwd_workspace_size", [ctypes.POINTER(BcastBwdArgs)], ctypes.c_size_t),
    ("jfa_decode_workspace_size", [ctypes.POINTER(DecodeArgs)], ctypes.c_size_t),
    ("jfa_varlen_fwd_workspace_size", [ctypes.POINTER(VarlenFwdArgs)], ctypes.c_size_t),
    ("jfa_varlen_bwd_workspace_size", [ctypes.POINTER(VarlenBwdArgs)], ctypes.c_size_t),
    ("jfa_decode_smallq_workspace_size", [ctypes.POINTER(DecodeSmallqArgs)], ctypes.c_size_t),
    ("jfa_fwd_fp8_workspace_size", [ctypes.POINTER(FwdFp8Args)], ctypes.c_size_t),
    ("jfa_fp8_quantize_v_workspace_size", [ctypes.POINTER(Fp8QuantizeVArgs)], ctypes.c_size_t),
    ("jfa_fp8_vt_bytes", [c_i32, c_i32, c_i32], ctypes.c_size_t),
    ("jfa_fwd", [ctypes.POINTER(FwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_bwd", [ctypes.POINTER(BwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_fwd_broadcast_q", [ctypes.POINTER(BcastFwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_bwd_broadcast_q", [ctypes.POINTER(BcastBwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_decode_splitkv", [ctypes.POINTER(DecodeArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_fwd_varlen", [ctypes.POINTER(VarlenFwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_bwd_varlen", [ctypes.POINTER(VarlenBwdArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_decode_smallq", [ctypes.POINTER(DecodeSmallqArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_fwd_fp8", [ctypes.POINTER(FwdFp8Args), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_fp8_quantize_v", [ctypes.POINTER(Fp8QuantizeVArgs), c_void_p, ctypes.c_size_t, c_void_p], c_i32),
    ("jfa_decode_splitkv_noalloc", [ctypes.POINTER(DecodeArgs), c_void_p], c_i32),
    ("jfa_decode_noalloc_status", [c_void_p, ctypes.POINTER(c_i32)], c_i32),
    ("jfa_read_device_status", [c_void_p, c_void_p, ctypes.POINTER(c_i32)], c_i32),
    ("jfa_selftest_wait_timeout", [c_i32, c_void_p, c_void_p], c_i32),
    ("jfa_trace_enable", [c_void_p, ctypes.c_size_t, c_i32], c_i32),
    ("jfa_trace_compiled", [], c_i32),
    ("jfa_status_string", [c_i32], ctypes.c_char_p),
    ("jfa_version", [], c_i32),
]

_lib = None


def load() -> ctypes.CDLL:
    """The loaded libjfa.so (or the variant JFA_LIBRARY_VARIANT names) with
    typed entry points. Raises if it is missing."""
    global _lib
    if _lib is None:
        variant = os.environ.get(VARIANT_ENV, "")
        if variant and variant not in ("trace", "debug"):
            raise RuntimeError(f"{VARIANT_ENV}={variant!r}: expected 'trace' or 'debug'")
        path = os.path.join(_PKG, f"libjfa_{variant}.so") if variant else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(or build.build(variant=...) for a debugging build; the CUDA library is required, "
                "there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, argtypes, restype in SIGNATURES:
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = lib
    return _lib
