"""Jagged (varlen) FlashAttention for GB300: Python binding of libjfa.so.

The functions here carry the names of the C entry points and only marshal
arguments: they check shapes and dtypes, allocate outputs and the workspace
with PyTorch when the caller does not pass them, and call the library on the
current CUDA stream. Every step of the computation runs in the sm_103a
kernels; there is no CPU or PyTorch fallback.

    jfa_fwd               jagged self-attention forward -> (O, LSE)
    jfa_bwd               its recompute-based backward -> (dQ, dK, dV)
    jfa_fwd_broadcast_q   one dense Q shared by a jagged K/V batch -> (O, LSE)
    jfa_bwd_broadcast_q   its backward, dQ summed over the batch -> (dQ, dK, dV)
    jfa_decode_splitkv    split-KV decode over a paged GQA cache -> (O, LSE)
    jfa_fwd_varlen        separate query / key lengths, grouped KV heads -> (O, LSE)
    jfa_bwd_varlen        its backward -> (dQ, dK, dV)
    jfa_decode_smallq     paged split-KV decode of a few query tokens per sequence -> (O, LSE)
    jfa_fwd_fp8           jagged forward over FP8 (e4m3) inputs with per-tensor descales -> (O, LSE)
    jfa_fp8_quantize_v    bf16 V -> e4m3 V in the layout jfa_fwd_fp8 reads (its vt argument)
    jfa_trace_enable      registers a per-role event trace buffer (JFA_TRACE builds; see trace.py)
    jfa_trace_compiled    1 if the loaded library records traces
    jagged_attention      autograd wrapper of jfa_fwd / jfa_bwd
    varlen_attention      autograd wrapper of jfa_fwd_varlen / jfa_bwd_varlen
"""
from __future__ import annotations

import contextlib
import ctypes
import math

import torch

from . import _abi

__all__ = [
    "JfaError", "jfa_fwd", "jfa_bwd", "jfa_fwd_broadcast_q", "jfa_bwd_broadcast_q", "jfa_decode_splitkv",
    "jfa_read_device_status", "jagged_attention", "library", "jfa_fwd_varlen", "jfa_bwd_varlen",
    "varlen_attention", "jfa_decode_smallq", "jfa_selftest_wait_timeout", "jfa_fwd_fp8",
    "jfa_trace_enable", "jfa_trace_compiled", "jfa_fp8_quantize_v",
]


class JfaError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = library().jfa_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def library():
    return _abi.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape):
    """Type, dtype, shape (a tuple, or an int: the number of dimensions) and
    layout of one argument. The kernels address every tensor from the shapes
    of q (and k), so each buffer is checked against them here; the device is
    checked by _device once every tensor of the call is known."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if isinstance(shape, int):
        if t.dim() != shape:
            raise ValueError(f"{name} must have {shape} dimensions, got {tuple(t.shape)}")
    elif t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_offsets(t, name):
    _need(t, name, torch.int32, 1)
    if t.numel() < 1:
        raise ValueError(f"{name} must hold batch + 1 >= 1 entries")


def _device(**tensors):
    """The one CUDA device that holds every given tensor (None entries are
    skipped); the call runs there, on that device's stream."""
    idx = None
    for name, t in tensors.items():
        if t is None:
            continue
        i = t.get_device()  # -1 on the host
        if i < 0:
            raise ValueError(f"{name} must be on a CUDA device")
        if idx is None:
            idx = i
        elif i != idx:
            raise ValueError(f"{name} is on cuda:{i}, the other tensors on cuda:{idx}")
    return torch.device("cuda", idx)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _events(events):
    if events is None:
        return None, None
    for e in events:  # torch creates the CUDA event lazily, on its first record
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * 2)(events[0].cuda_event, events[1].cuda_event)
    return ctypes.cast(arr, ctypes.c_void_p), arr


def _workspace(nbytes, device, workspace):
    if workspace is None:
        return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor")
    if workspace.get_device() != device.index:
        raise ValueError(f"workspace is on {workspace.device}, the call runs on {device}")
    if _nbytes(workspace) < nbytes:
        raise ValueError(f"workspace holds {_nbytes(workspace)} bytes, needs {nbytes}")
    return workspace


def _nbytes(t):
    return t.numel() * t.element_size()


def _run(entry, size_entry, a, device, workspace, stream, check):
    """Sizes the workspace, calls the entry point on `device` and its stream,
    and with check=True reads the device status back (a stream sync)."""
    lib = library()
    here = device.index == torch.cuda.current_device()
    with contextlib.nullcontext() if here else torch.cuda.device(device):
        if stream is not None and stream.device_index != device.index:
            raise ValueError(f"stream belongs to {stream.device}, the call runs on {device}")
        ws = _workspace(getattr(lib, size_entry)(ctypes.byref(a)), device, workspace)
        _check(getattr(lib, entry)(ctypes.byref(a), _ptr(ws), _nbytes(ws), _stream(stream)), entry)
        _finish(ws, check, stream, entry)


def _check(status, where):
    if status != _abi.JFA_OK:
        raise JfaError(status, where)


def jfa_read_device_status(workspace, stream=None):
    """Synchronises the stream; returns (status, detail) of the last call that used `workspace`."""
    d = ctypes.c_int32(0)
    st = library().jfa_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(d))
    return int(st), int(d.value)


def jfa_selftest_wait_timeout(budget_us=20000, workspace=None, stream=None):
    """Runs the failure-detection self-test (a pipeline wait whose input never
    arrives, bounded to budget_us). Returns (status, detail, second_stage_aborted)."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda") if workspace is None else workspace
    _check(library().jfa_selftest_wait_timeout(int(budget_us), _ptr(ws), _stream(stream)), "jfa_selftest_wait_timeout")
    st, detail = jfa_read_device_status(ws, stream)
    aborted = int(ws[16:20].view(torch.int32).item())
    return st, detail, aborted


def jfa_trace_compiled():
    """1 if the loaded library was built with JFA_TRACE (it records traces), else 0."""
    return int(library().jfa_trace_compiled())


def jfa_trace_enable(buffer, records_per_warp=1024):
    """Registers `buffer` (a zeroed uint8 CUDA tensor of at least
    trace.buffer_bytes(SMs, records_per_warp) bytes) for the per-role event
    records of later calls; None turns recording off. Raises JfaError
    (unsupported) unless the library was built with JFA_TRACE."""
    if buffer is not None:
        if not isinstance(buffer, torch.Tensor) or not buffer.is_cuda or not buffer.is_contiguous():
            raise TypeError("buffer must be a contiguous CUDA tensor")
        _check(library().jfa_trace_enable(_ptr(buffer), _nbytes(buffer), int(records_per_warp)), "jfa_trace_enable")
    else:
        _check(library().jfa_trace_enable(None, 0, 0), "jfa_trace_enable")


def _finish(ws, check, stream, where):
    if check:
        st, detail = jfa_read_device_status(ws, stream)
        if st != _abi.JFA_OK:
            e = JfaError(st, f"{where} (device, detail {detail})")
            raise e


# ---------------------------------------------------------------- forward / backward

def jfa_fwd(q, k, v, offsets, max_seqlen, scale=None, causal=False, o=None, lse=None, workspace=None,
            stream=None, events=None, check=False):
    """Jagged self-attention forward. q, k, v: bf16 [total, H, d]; offsets: int32 [B+1] (CUDA).
    Returns O bf16 [total, H, d] and LSE fp32 [H, total] (natural log)."""
    _need(q, "q", torch.bfloat16, 3)
    total, H, d = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need_offsets(offsets, "offsets")
    if o is not None:
        _need(o, "o", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (H, total))
    dev = _device(q=q, k=k, v=v, offsets=offsets, o=o, lse=lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((H, total), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.FwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), offsets.numel() - 1, H, d, int(max_seqlen),
                     total, scale, int(bool(causal)), _ptr(o), _ptr(lse), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_fwd", "jfa_fwd_workspace_size", a, dev, workspace, stream, check)
    return o, lse


def jfa_bwd(q, k, v, o, dout, lse, offsets, max_seqlen, scale=None, causal=False, head_chunk=0,
            dq=None, dk=None, dv=None, workspace=None, stream=None, events=None, check=False):
    """Recompute-based backward of jfa_fwd. Returns dQ, dK, dV bf16 [total, H, d]."""
    _need(q, "q", torch.bfloat16, 3)
    total, H, d = q.shape
    for n, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need(t, n, torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (H, total))
    _need_offsets(offsets, "offsets")
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t is not None:
            _need(t, n, torch.bfloat16, q.shape)
    dev = _device(q=q, k=k, v=v, o=o, dout=dout, lse=lse, offsets=offsets, dq=dq, dk=dk, dv=dv)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    a = _abi.BwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(offsets),
                     offsets.numel() - 1, H, d, int(max_seqlen), total, scale, int(bool(causal)), int(head_chunk),
                     _ptr(dq), _ptr(dk), _ptr(dv), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_bwd", "jfa_bwd_workspace_size", a, dev, workspace, stream, check)
    return dq, dk, dv


def jfa_fwd_broadcast_q(q, k, v, kv_offsets, max_seqlen_k, scale=None, o=None, lse=None, workspace=None,
                        stream=None, events=None, check=False):
    """Broadcast-Q forward. q: bf16 [Lq, H, d] shared by every sequence; k, v jagged [total_k, H, d].
    Returns O bf16 [B, Lq, H, d] and LSE fp32 [B, H, Lq]."""
    _need(q, "q", torch.bfloat16, 3)
    Lq, H, d = q.shape
    _need(k, "k", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, (k.shape[0], H, d))
    _need(v, "v", torch.bfloat16, k.shape)
    _need_offsets(kv_offsets, "kv_offsets")
    B = kv_offsets.numel() - 1
    if o is not None:
        _need(o, "o", torch.bfloat16, (B, Lq, H, d))
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, Lq))
    dev = _device(q=q, k=k, v=v, kv_offsets=kv_offsets, o=o, lse=lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((B, Lq, H, d), dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.BcastFwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(kv_offsets), B, Lq, H, d, int(max_seqlen_k),
                          k.shape[0], scale, _ptr(o), _ptr(lse), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_fwd_broadcast_q", "jfa_bcast_fwd_workspace_size", a, dev, workspace, stream, check)
    return o, lse


def jfa_bwd_broadcast_q(q, k, v, o, dout, lse, kv_offsets, max_seqlen_k, scale=None, dq=None, dk=None, dv=None,
                        workspace=None, stream=None, events=None, check=False):
    """Broadcast-Q backward. Returns dQ bf16 [Lq, H, d] summed over the batch, dK, dV [total_k, H, d]."""
    _need(q, "q", torch.bfloat16, 3)
    Lq, H, d = q.shape
    _need(k, "k", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, (k.shape[0], H, d))
    _need(v, "v", torch.bfloat16, k.shape)
    _need_offsets(kv_offsets, "kv_offsets")
    B = kv_offsets.numel() - 1
    _need(o, "o", torch.bfloat16, (B, Lq, H, d))
    _need(dout, "dout", torch.bfloat16, (B, Lq, H, d))
    _need(lse, "lse", torch.float32, (B, H, Lq))
    if dq is not None:
        _need(dq, "dq", torch.bfloat16, q.shape)
    if dk is not None:
        _need(dk, "dk", torch.bfloat16, k.shape)
    if dv is not None:
        _need(dv, "dv", torch.bfloat16, k.shape)
    dev = _device(q=q, k=k, v=v, o=o, dout=dout, lse=lse, kv_offsets=kv_offsets, dq=dq, dk=dk, dv=dv)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    a = _abi.BcastBwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(kv_offsets),
                          B, Lq, H, d, int(max_seqlen_k), k.shape[0], scale, _ptr(dq), _ptr(dk), _ptr(dv), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_bwd_broadcast_q", "jfa_bcast_bwd_workspace_size", a, dev, workspace, stream, check)
    return dq, dk, dv


def jfa_fwd_fp8(q, k, v, offsets, max_seqlen, q_descale, k_descale, v_descale, scale=None, causal=False, o=None,
                lse=None, workspace=None, stream=None, events=None, check=False, vt=None):
    """Jagged forward over FP8 inputs. q, k, v: e4m3 codes [total, H, 128] (torch.uint8 or
    torch.float8_e4m3fn); byte x of q stands for e4m3(x) * q_descale (likewise k, v).
    vt (optional): V as jfa_fp8_quantize_v wrote it for these offsets and heads; v is then
    not read (it may be None) and the call makes no pass over V.
    Returns O bf16 [total, H, 128] and LSE fp32 [H, total]."""
    qkv = []
    for n, t in (("q", q), ("k", k), ("v", v)):
        if n == "v" and t is None and vt is not None:
            qkv.append(None)
            continue
        if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        _need(t, n, torch.uint8, 3)
        qkv.append(t)
    q, k, v = qkv
    total, H, d = q.shape
    _need(k, "k", torch.uint8, q.shape)
    if v is not None:
        _need(v, "v", torch.uint8, q.shape)
    _need_offsets(offsets, "offsets")
    if vt is not None:
        _need(vt, "vt", torch.uint8, (int(library().jfa_fp8_vt_bytes(offsets.numel() - 1, H, total)),))
    if o is not None:
        _need(o, "o", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (H, total))
    dev = _device(q=q, k=k, v=v, offsets=offsets, o=o, lse=lse, vt=vt)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((total, H, d), dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty((H, total), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.FwdFp8Args(_ptr(q), _ptr(k), _ptr(v), _ptr(offsets), offsets.numel() - 1, H, d, int(max_seqlen), total,
                        scale, int(bool(causal)), float(q_descale), float(k_descale), float(v_descale), _ptr(o),
                        _ptr(lse), None, _ptr(vt))
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_fwd_fp8", "jfa_fwd_fp8_workspace_size", a, dev, workspace, stream, check)
    return o, lse


def jfa_fp8_quantize_v(v, offsets, max_seqlen, v_descale, vt=None, workspace=None, stream=None, check=False):
    """bf16 V [total, H, 128] -> e4m3(v / v_descale) in the blocks jfa_fwd_fp8 reads (see
    include/jfa.h): returns the uint8 tensor of jfa_fp8_vt_bytes(batch, H, total) bytes, to
    pass as jfa_fwd_fp8(..., vt=...)."""
    _need(v, "v", torch.bfloat16, 3)
    total, H, d = v.shape
    _need_offsets(offsets, "offsets")
    nbytes = int(library().jfa_fp8_vt_bytes(offsets.numel() - 1, H, total))
    if vt is not None:
        _need(vt, "vt", torch.uint8, (nbytes,))
    dev = _device(v=v, offsets=offsets, vt=vt)
    vt = torch.empty(nbytes, dtype=torch.uint8, device=dev) if vt is None else vt
    a = _abi.Fp8QuantizeVArgs(_ptr(v), _ptr(offsets), offsets.numel() - 1, H, d, int(max_seqlen), total,
                              float(v_descale), _ptr(vt))
    _run("jfa_fp8_quantize_v", "jfa_fp8_quantize_v_workspace_size", a, dev, workspace, stream, check)
    return vt


# ---------------------------------------------------------------- varlen / GQA

def _var_inputs(q, k, v, q_offsets, k_offsets):
    _need(q, "q", torch.bfloat16, 3)
    total_q, Hq, d = q.shape
    _need(k, "k", torch.bfloat16, 3)
    total_k, Hkv, _ = k.shape
    _need(k, "k", torch.bfloat16, (total_k, Hkv, d))
    _need(v, "v", torch.bfloat16, k.shape)
    _need_offsets(q_offsets, "q_offsets")
    _need_offsets(k_offsets, "k_offsets")
    if q_offsets.numel() != k_offsets.numel():
        raise ValueError("q_offsets and k_offsets must have the same length")
    return total_q, Hq, d, total_k, Hkv


def jfa_fwd_varlen(q, k, v, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale=None, causal=False, o=None,
                   lse=None, workspace=None, stream=None, events=None, check=False):
    """Jagged attention with separate query / key packing and grouped KV heads.
    q: bf16 [total_q, Hq, d]; k, v: bf16 [total_k, Hkv, d] with Hq % Hkv == 0; q_offsets and
    k_offsets: int32 [B+1] (CUDA). causal aligns the mask to the bottom right (key j visible to
    query i iff j <= i + L_k - L_q). Returns O bf16 [total_q, Hq, d], LSE fp32 [Hq, total_q]."""
    total_q, Hq, d, total_k, Hkv = _var_inputs(q, k, v, q_offsets, k_offsets)
    if o is not None:
        _need(o, "o", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (Hq, total_q))
    dev = _device(q=q, k=k, v=v, q_offsets=q_offsets, k_offsets=k_offsets, o=o, lse=lse)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((Hq, total_q), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.VarlenFwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(q_offsets), _ptr(k_offsets), q_offsets.numel() - 1,
                           Hq, Hkv, d, int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, scale,
                           int(bool(causal)), _ptr(o), _ptr(lse), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_fwd_varlen", "jfa_varlen_fwd_workspace_size", a, dev, workspace, stream, check)
    return o, lse


def jfa_bwd_varlen(q, k, v, o, dout, lse, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale=None,
                   causal=False, head_chunk=0, dq=None, dk=None, dv=None, workspace=None, stream=None, events=None,
                   check=False):
    """Backward of jfa_fwd_varlen. Returns dQ bf16 [total_q, Hq, d] and dK, dV bf16
    [total_k, Hkv, d] (a KV head's gradient summed over the query heads that read it)."""
    total_q, Hq, d, total_k, Hkv = _var_inputs(q, k, v, q_offsets, k_offsets)
    _need(o, "o", torch.bfloat16, q.shape)
    _need(dout, "dout", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (Hq, total_q))
    if dq is not None:
        _need(dq, "dq", torch.bfloat16, q.shape)
    if dk is not None:
        _need(dk, "dk", torch.bfloat16, k.shape)
    if dv is not None:
        _need(dv, "dv", torch.bfloat16, k.shape)
    dev = _device(q=q, k=k, v=v, o=o, dout=dout, lse=lse, q_offsets=q_offsets, k_offsets=k_offsets, dq=dq, dk=dk,
                  dv=dv)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    a = _abi.VarlenBwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(q_offsets),
                           _ptr(k_offsets), q_offsets.numel() - 1, Hq, Hkv, d, int(max_seqlen_q), int(max_seqlen_k),
                           total_q, total_k, scale, int(bool(causal)), int(head_chunk), _ptr(dq), _ptr(dk), _ptr(dv),
                           None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_bwd_varlen", "jfa_varlen_bwd_workspace_size", a, dev, workspace, stream, check)
    return dq, dk, dv


# ---------------------------------------------------------------- decode

def _cache_inputs(k_cache, v_cache, page_table, seqlens_k, B, d):
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    num_pages, P, Hkv, _ = k_cache.shape
    _need(k_cache, "k_cache", torch.bfloat16, (num_pages, P, Hkv, d))
    _need(v_cache, "v_cache", torch.bfloat16, k_cache.shape)
    _need(page_table, "page_table", torch.int32, 2)
    _need(page_table, "page_table", torch.int32, (B, page_table.shape[1]))
    _need(seqlens_k, "seqlens_k", torch.int32, (B,))
    return num_pages, P, Hkv


def jfa_decode_splitkv(q, k_cache, v_cache, page_table, seqlens_k, num_splits, scale=None, o=None, lse=None,
                       split_bounds=None, workspace=None, stream=None, events=None, check=False):
    """Split-KV decode over a paged GQA cache. q: bf16 [B, Hq, 128]; caches bf16
    [num_pages, page_size, Hkv, 128]; page_table int32 [B, max_pages]; seqlens_k int32 [B].
    Returns O bf16 [B, Hq, 128] and LSE fp32 [B, Hq]. If `split_bounds` (int32 [B, S, 2])
    is given, the kernel writes each split's token range into it."""
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, d = q.shape
    num_pages, P, Hkv = _cache_inputs(k_cache, v_cache, page_table, seqlens_k, B, d)
    if split_bounds is not None:
        _need(split_bounds, "split_bounds", torch.int32, (B, int(num_splits), 2))
    if o is not None:
        _need(o, "o", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, Hq))
    dev = _device(q=q, k_cache=k_cache, v_cache=v_cache, page_table=page_table, seqlens_k=seqlens_k, o=o, lse=lse,
                  split_bounds=split_bounds)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.DecodeArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seqlens_k),
                        B, Hq, Hkv, d, P, num_pages, page_table.shape[1], int(num_splits), scale,
                        _ptr(o), _ptr(lse), _ptr(split_bounds), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_decode_splitkv", "jfa_decode_workspace_size", a, dev, workspace, stream, check)
    return o, lse


def jfa_decode_smallq(q, k_cache, v_cache, page_table, seqlens_k, num_splits, min_split_tokens=0, scale=None,
                      o=None, lse=None, split_bounds=None, split_counts=None, workspace=None, stream=None,
                      events=None, check=False):
    """Paged split-KV decode of q_len new tokens per sequence (speculative / chunked decode).
    q: bf16 [B, q_len, Hq, 128]; caches bf16 [num_pages, page_size, Hkv, 128]; page_table int32
    [B, max_pages]; seqlens_k int32 [B] (new tokens included: token i of q_len sits at key position
    L - q_len + i and sees keys up to it). Returns O bf16 [B, q_len, Hq, 128], LSE fp32 [B, q_len, Hq].
    With min_split_tokens > 0 each sequence uses clamp(ceil(L / min_split_tokens), 1, num_splits)
    splits; `split_counts` (int32 [B]) and `split_bounds` (int32 [B, S, 2]) receive them if given."""
    _need(q, "q", torch.bfloat16, 4)
    B, ql, Hq, d = q.shape
    num_pages, P, Hkv = _cache_inputs(k_cache, v_cache, page_table, seqlens_k, B, d)
    if split_bounds is not None:
        _need(split_bounds, "split_bounds", torch.int32, (B, int(num_splits), 2))
    if split_counts is not None:
        _need(split_counts, "split_counts", torch.int32, (B,))
    if o is not None:
        _need(o, "o", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, ql, Hq))
    dev = _device(q=q, k_cache=k_cache, v_cache=v_cache, page_table=page_table, seqlens_k=seqlens_k, o=o, lse=lse,
                  split_bounds=split_bounds, split_counts=split_counts)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, ql, Hq), dtype=torch.float32, device=dev) if lse is None else lse
    a = _abi.DecodeSmallqArgs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seqlens_k),
                              B, ql, Hq, Hkv, d, P, num_pages, page_table.shape[1], int(num_splits),
                              int(min_split_tokens), scale, _ptr(o), _ptr(lse), _ptr(split_bounds),
                              _ptr(split_counts), None)
    ev, _keep = _events(events)
    a.main_kernel_events = ev
    _run("jfa_decode_smallq", "jfa_decode_smallq_workspace_size", a, dev, workspace, stream, check)
    return o, lse


# ---------------------------------------------------------------- autograd

class _JaggedAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, offsets, max_seqlen, scale, causal):
        o, lse = jfa_fwd(q, k, v, offsets, max_seqlen, scale, causal)
        ctx.save_for_backward(q, k, v, o, lse, offsets)
        ctx.max_seqlen, ctx.scale, ctx.causal = max_seqlen, scale, causal
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, offsets = ctx.saved_tensors
        dq, dk, dv = jfa_bwd(q, k, v, o, do.contiguous(), lse, offsets, ctx.max_seqlen, ctx.scale, ctx.causal)
        return dq, dk, dv, None, None, None, None


def jagged_attention(q, k, v, offsets, max_seqlen, scale=None, causal=False):
    """Differentiable jagged attention (bf16 [total, H, d] tensors, int32 offsets)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _JaggedAttention.apply(q, k, v, offsets, max_seqlen, scale, causal)


class _VarlenAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale, causal):
        o, lse = jfa_fwd_varlen(q, k, v, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale, causal)
        ctx.save_for_backward(q, k, v, o, lse, q_offsets, k_offsets)
        ctx.args = (max_seqlen_q, max_seqlen_k, scale, causal)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, q_offsets, k_offsets = ctx.saved_tensors
        mq, mk, scale, causal = ctx.args
        dq, dk, dv = jfa_bwd_varlen(q, k, v, o, do.contiguous(), lse, q_offsets, k_offsets, mq, mk, scale, causal)
        return dq, dk, dv, None, None, None, None, None, None


def varlen_attention(q, k, v, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale=None, causal=False):
    """Differentiable varlen / GQA attention (see jfa_fwd_varlen for layouts and the causal alignment)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _VarlenAttention.apply(q, k, v, q_offsets, k_offsets, max_seqlen_q, max_seqlen_k, scale, causal)
