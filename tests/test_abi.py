"""The C ABI on the CPU: the library loads without a GPU, exports every symbol
include/jfa.h declares, the ctypes structures match the C layout (checked
against a C program compiled with the header), and host-side validation
rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import varlen_flashattention_gb300 as jfa
from varlen_flashattention_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jfa.h")
CUDA_INC = "/usr/local/cuda/include"

STRUCTS = {
    "jfa_fwd_args": _abi.FwdArgs,
    "jfa_bwd_args": _abi.BwdArgs,
    "jfa_bcast_fwd_args": _abi.BcastFwdArgs,
    "jfa_bcast_bwd_args": _abi.BcastBwdArgs,
    "jfa_decode_args": _abi.DecodeArgs,
    "jfa_varlen_fwd_args": _abi.VarlenFwdArgs,
    "jfa_varlen_bwd_args": _abi.VarlenBwdArgs,
    "jfa_decode_smallq_args": _abi.DecodeSmallqArgs,
    "jfa_fwd_fp8_args": _abi.FwdFp8Args,
    "jfa_fp8_quantize_v_args": _abi.Fp8QuantizeVArgs,
}


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"JFA_API\s+[\w\s\*]+?\b(jfa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from __graft_entry__ import build
    build()
    return jfa.library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 13, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in jfa.h but not exported"
    assert {s[0] for s in _abi.SIGNATURES} == set(names)


def test_struct_layouts_match_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime_api.h")):
        pytest.skip("gcc or CUDA headers missing")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "jfa.h"', "int main(void) {"]
    for cname, py in STRUCTS.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call([gcc, "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    got = {}
    for line in out:
        if line:
            s, f, v = line.split()
            got[(s, f)] = int(v)
    for cname, py in STRUCTS.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_status_strings(lib):
    for code in range(7):
        assert lib.jfa_status_string(code)
    assert lib.jfa_version() >= 100


FAKE = 0x10000  # aligned, never dereferenced: every call below returns before any CUDA work


def _fwd_args(**kw):
    a = _abi.FwdArgs(FAKE, FAKE, FAKE, FAKE, 2, 4, 128, 100, 150, 0.1, 0, FAKE, FAKE, None)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_fwd_validation(lib):
    P = ctypes.byref
    assert lib.jfa_fwd(None, FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_fwd(P(_fwd_args(head_dim=96)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_fwd(P(_fwd_args(q=FAKE + 8)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_fwd(P(_fwd_args(scale=-1.0)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_fwd(P(_fwd_args(causal=2)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_fwd(P(_fwd_args(heads=0)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_fwd(P(_fwd_args()), FAKE + 16, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG  # ws alignment
    need = lib.jfa_fwd_workspace_size(P(_fwd_args()))
    assert need > 256
    assert lib.jfa_fwd(P(_fwd_args()), FAKE, need - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_bwd_validation(lib):
    P = ctypes.byref

    def args(**kw):
        a = _abi.BwdArgs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 128, 100, 150, 0.1, 0, 0, FAKE, FAKE, FAKE,
                         None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    assert lib.jfa_bwd(P(args(head_dim=192, head_chunk=192)), FAKE, 1 << 40, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_bwd(P(args(head_dim=64, head_chunk=32)), FAKE, 1 << 40, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_bwd(P(args(dq=FAKE + 4)), FAKE, 1 << 40, None) == _abi.JFA_ERR_INVALID_ARG
    need = lib.jfa_bwd_workspace_size(P(args()))
    # the fp32 dQ accumulator dominates: total * heads * head_dim * 4 bytes
    assert need >= 150 * 4 * 128 * 4
    assert lib.jfa_bwd(P(args()), FAKE, need - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_decode_validation(lib):
    P = ctypes.byref

    def args(**kw):
        a = _abi.DecodeArgs(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 32, 8, 128, 16, 100, 10, 8, 0.1, FAKE, FAKE, None, None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    for bad in (dict(num_splits=0), dict(num_splits=129), dict(page_size=0), dict(q_heads=30),
                dict(seqlens_k=FAKE + 2)):
        assert lib.jfa_decode_splitkv(P(args(**bad)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG, bad
    assert lib.jfa_decode_splitkv(P(args(head_dim=64)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_decode_splitkv(P(args(kv_heads=1)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED  # group 32
    need = lib.jfa_decode_workspace_size(P(args()))
    assert need >= 8 * 4 * 32 * 128 * 4
    assert lib.jfa_decode_splitkv(P(args()), FAKE, need - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_decode_noalloc_validation_precedes_the_size_limit(lib):
    """A malformed request to the allocation-free decode is refused as such,
    not as one too large for its scratch (the checks run before the limit)."""
    P = ctypes.byref

    def args(**kw):
        a = _abi.DecodeArgs(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 32, 8, 128, 16, 100, 10, 8, 0.1, FAKE, FAKE, None, None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    assert lib.jfa_decode_splitkv_noalloc(None, None) == _abi.JFA_ERR_INVALID_ARG
    # num_splits 129 with a batch that would also overflow the 32768-row scratch
    for bad in (dict(batch=-1), dict(num_splits=129), dict(num_splits=129, batch=64), dict(num_splits=0),
                dict(page_size=0), dict(q=FAKE + 8)):
        assert lib.jfa_decode_splitkv_noalloc(P(args(**bad)), None) == _abi.JFA_ERR_INVALID_ARG, bad
    assert lib.jfa_decode_splitkv_noalloc(P(args(head_dim=64)), None) == _abi.JFA_ERR_UNSUPPORTED
    # a well-formed request above the limit: 32 splits x 64 sequences x 32 heads = 65536 rows
    assert lib.jfa_decode_splitkv_noalloc(P(args(batch=64, num_splits=32)), None) == \
        _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_varlen_validation(lib):
    P = ctypes.byref

    def fargs(**kw):
        a = _abi.VarlenFwdArgs(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 100, 300, 150, 400, 0.1, 1,
                               FAKE, FAKE, None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    def bargs(**kw):
        a = _abi.VarlenBwdArgs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 100, 300, 150, 400,
                               0.1, 1, 0, FAKE, FAKE, FAKE, None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    for bad in (dict(kv_heads=3), dict(kv_heads=0), dict(k_offsets=FAKE + 2), dict(k=FAKE + 8), dict(causal=2),
                dict(total_k=-1)):
        assert lib.jfa_fwd_varlen(P(fargs(**bad)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG, bad
        assert lib.jfa_bwd_varlen(P(bargs(**bad)), FAKE, 1 << 40, None) == _abi.JFA_ERR_INVALID_ARG, bad
    assert lib.jfa_fwd_varlen(P(fargs(head_dim=96)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_bwd_varlen(P(bargs(head_dim=192, head_chunk=192)), FAKE, 1 << 40, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_bwd_varlen(P(bargs(dk=FAKE + 4)), FAKE, 1 << 40, None) == _abi.JFA_ERR_INVALID_ARG
    # forward items: query tiles of every query head; backward: key tiles of every KV head,
    # plus the fp32 dQ accumulator over the queries
    nf = lib.jfa_varlen_fwd_workspace_size(P(fargs()))
    assert nf >= 256 + 2 * 16 * 8 * (2 + 2)
    nb = lib.jfa_varlen_bwd_workspace_size(P(bargs()))
    assert nb >= 150 * 8 * 128 * 4
    assert lib.jfa_fwd_varlen(P(fargs()), FAKE, nf - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL
    assert lib.jfa_bwd_varlen(P(bargs()), FAKE, nb - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_decode_smallq_validation(lib):
    P = ctypes.byref

    def args(**kw):
        a = _abi.DecodeSmallqArgs(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 32, 8, 128, 16, 100, 10, 8, 0, 0.1,
                                  FAKE, FAKE, None, None, None)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    for bad in (dict(q_len=0), dict(num_splits=0), dict(min_split_tokens=-1), dict(q_heads=30),
                dict(split_counts_out=FAKE + 2)):
        assert lib.jfa_decode_smallq(P(args(**bad)), FAKE, 1 << 30, None) == _abi.JFA_ERR_INVALID_ARG, bad
    # the (token, head) rows of one KV head must fit one 16-row tile
    assert lib.jfa_decode_smallq(P(args(q_len=5)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED
    assert lib.jfa_decode_smallq(P(args(head_dim=64)), FAKE, 1 << 30, None) == _abi.JFA_ERR_UNSUPPORTED
    need = lib.jfa_decode_smallq_workspace_size(P(args()))
    assert need >= 8 * 4 * 4 * 32 * 128 * 4
    assert lib.jfa_decode_smallq(P(args()), FAKE, need - 1, None) == _abi.JFA_ERR_WORKSPACE_TOO_SMALL


def test_selftest_validation(lib):
    assert lib.jfa_selftest_wait_timeout(0, FAKE, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_selftest_wait_timeout(10 ** 8, FAKE, None) == _abi.JFA_ERR_INVALID_ARG
    assert lib.jfa_selftest_wait_timeout(1000, FAKE + 16, None) == _abi.JFA_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        jfa.jfa_fwd(q, q, q, torch.zeros(2, dtype=torch.int32), 4)


def test_trace_entry_points_of_the_default_build(lib):
    assert lib.jfa_trace_compiled() == 0
    assert lib.jfa_trace_enable(None, 0, 0) == _abi.JFA_ERR_UNSUPPORTED
    with pytest.raises(jfa.JfaError):
        jfa.jfa_trace_enable(None)


_VARIANT_PROBE = r"""
import ctypes, sys
from varlen_flashattention_gb300 import _abi
lib = _abi.load()
assert lib._name.endswith("libjfa_%s.so" % sys.argv[1]), lib._name
print(lib.jfa_trace_compiled(), lib.jfa_trace_enable(None, 0, 0), lib.jfa_trace_enable(ctypes.c_void_p(4096), 16, 0))
"""


@pytest.mark.parametrize("variant", ["trace", "debug"])
def test_debugging_builds_compile_and_export_the_abi(variant):
    """Each debugging build compiles, loads in place of libjfa.so when JFA_LIBRARY_VARIANT names
    it, exports every declared symbol, and answers the trace entry points for its build."""
    from varlen_flashattention_gb300 import build
    path = build.build(variant=variant)
    vlib = ctypes.CDLL(path)
    for n in _declared_functions():
        assert hasattr(vlib, n), f"{n} not exported by {os.path.basename(path)}"
    env = dict(os.environ, JFA_LIBRARY_VARIANT=variant)
    r = subprocess.run(["python", "-c", _VARIANT_PROBE, variant], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    compiled, off, bad = (int(x) for x in r.stdout.split())
    if variant == "trace":
        assert (compiled, off, bad) == (1, _abi.JFA_OK, _abi.JFA_ERR_INVALID_ARG)
    else:
        assert (compiled, off, bad) == (0, _abi.JFA_ERR_UNSUPPORTED, _abi.JFA_ERR_UNSUPPORTED)


def test_fp8_quantize_v_validation(lib):
    """jfa_fp8_quantize_v checks its arguments on the host; jfa_fp8_vt_bytes sizes the blocks."""
    assert lib.jfa_fp8_vt_bytes(3, 2, 300) == (3 + 3) * 2 * 16384  # ceil(300/128) + batch tiles per head
    assert lib.jfa_fp8_vt_bytes(-1, 2, 300) == 0 and lib.jfa_fp8_vt_bytes(3, 0, 300) == 0
    ok = dict(v=None, offsets=None, batch=0, heads=2, head_dim=128, max_seqlen=0, total=0, v_descale=1.0, vt=None)
    ws = ctypes.c_void_p(256)
    assert lib.jfa_fp8_quantize_v(ctypes.byref(_abi.Fp8QuantizeVArgs(**{**ok, "head_dim": 64})), ws, 4096,
                                  None) == _abi.JFA_ERR_UNSUPPORTED
    for bad in ({"v_descale": 0.0}, {"v_descale": float("inf")}, {"v_descale": 1e-45}, {"batch": -1},
                {"heads": 0}, {"total": -1}):
        a = _abi.Fp8QuantizeVArgs(**{**ok, **bad})
        assert lib.jfa_fp8_quantize_v(ctypes.byref(a), ws, 4096, None) == _abi.JFA_ERR_INVALID_ARG, bad
    assert lib.jfa_fp8_quantize_v(None, ws, 4096, None) == _abi.JFA_ERR_INVALID_ARG
