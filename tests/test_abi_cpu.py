"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching the GPU.

No compute call is made: every call here fails validation, which happens on
the host before anything is enqueued, so fake (never dereferenced) device
addresses are safe to pass.
"""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_gb300 as kda
from kimi_delta_attention_gb300 import _lib
from kimi_delta_attention_gb300.builder import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load_library()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_exports_match_header(lib):
    declared = header_symbols()
    assert declared == sorted(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(10):
        s = kda.kda_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert kda.kda_status_string(99) == "unknown status"


def test_workspace_size_and_chunk(lib):
    shape = _lib.KdaShape(1, 4096, 32, 32, 128, 128, 0, _lib.KDA_BF16)
    assert kda.kda_chunk_fwd_workspace_size(shape) >= 256
    assert kda.kda_chunk_size() in (16, 32, 64, 128)


def test_kernel_name_query(lib):
    """Host-only: names the kernel a shape dispatches to (no GPU needed)."""
    f32 = _lib.KdaShape(1, 128, 2, 2, 64, 64, 0, _lib.KDA_F32)
    assert kda.kda_chunk_fwd_kernel_name(f32) == "recurrent_fwd_kernel"
    bf16 = _lib.KdaShape(1, 4096, 32, 32, 128, 128, 0, _lib.KDA_BF16)
    assert kda.kda_chunk_fwd_kernel_name(bf16) in ("kda_chunk_split_kernel", "kda_chunk_fused_kernel",
                                                   "recurrent_fwd_kernel")
    empty = _lib.KdaShape(1, 0, 2, 2, 128, 128, 0, _lib.KDA_BF16)
    assert kda.kda_chunk_fwd_kernel_name(empty) == "none"
    assert lib.kda_chunk_fwd_kernel_name(None) == b"none"
    assert kda.kda_chunk_fwd_kernel_launches(f32) == 1
    assert kda.kda_chunk_fwd_kernel_launches(empty) == 0
    assert lib.kda_chunk_fwd_kernel_launches(None) == 0


FAKE = 0x10000  # aligned, never dereferenced


def call(lib, shape, q=FAKE, k=FAKE + 0x100000, v=FAKE + 0x200000, g=FAKE + 0x300000,
         beta=FAKE + 0x400000, scale=0.088, s0=None, cu=None, out=FAKE + 0x500000,
         sfin=None, ws=FAKE + 0x600000, ws_bytes=256, entry="kda_chunk_fwd"):
    P = ctypes.c_void_p
    return getattr(lib, entry)(ctypes.byref(shape), P(q), P(k), P(v), P(g), P(beta), ctypes.c_float(scale),
                               P(s0), P(cu), P(out), P(sfin), P(ws), ctypes.c_size_t(ws_bytes), P(0))


def S(B=1, T=8, H=2, HV=2, K=64, V=64, ns=0, io=_lib.KDA_F32):
    return _lib.KdaShape(B, T, H, HV, K, V, ns, io)


@pytest.mark.parametrize("entry", ["kda_chunk_fwd", "kda_recurrent_fwd"])
def test_host_validation_rejects(lib, entry):
    c = lambda *a, **kw: call(lib, *a, entry=entry, **kw)
    assert c(S(HV=3, H=2)) == 1                       # HV % H != 0
    assert c(S(H=0)) == 1
    assert c(S(T=-1)) == 1
    assert c(S(K=96)) == 2                            # unsupported head dim
    assert c(S(V=32)) == 2
    assert c(S(io=5)) == 1                            # bad dtype
    assert c(S(), scale=0.0) == 1
    assert c(S(), scale=float("nan")) == 1
    assert c(S(), q=None) == 1                        # null required pointer
    assert c(S(), out=None) == 1
    assert c(S(), q=FAKE + 8) == 3                    # misaligned
    assert c(S(), g=FAKE + 0x300000 + 4) == 3
    assert c(S(), beta=FAKE + 0x400000 + 2) == 3
    assert c(S(), ws=None) == 6                       # workspace missing
    assert c(S(), ws_bytes=16) == 6                   # workspace too small
    assert c(S(B=2, ns=1), cu=FAKE + 0x700000) == 1   # varlen needs B == 1
    assert c(S(ns=0), cu=FAKE + 0x700000) == 1        # varlen needs num_seqs >= 1
    assert c(S(ns=2)) == 1                            # num_seqs without cu_seqlens
    assert c(S(), out=FAKE) == 1                      # out aliases q
    assert c(S(), sfin=FAKE + 0x300000) == 1          # final state aliases g
    assert c(S(), s0=FAKE + 0x800000, sfin=FAKE + 0x800000 + 16) == 1  # partial overlap


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        _lib.load_library(str(tmp_path / "nope.so"))


def test_binding_refuses_host_tensors(lib):
    """The binding has no CPU path: host tensors are refused before any call."""
    import torch
    from kimi_delta_attention_gb300 import workloads as W
    x = W.make_inputs(1, 64, 1, 1, 128, 128, "bf16", seed=1)
    for fn in (kda.kda_chunk_fwd, kda.kda_recurrent_fwd):
        with pytest.raises(_lib.KdaError):
            fn(x.q, x.k, x.v, x.g, x.beta, x.scale)
    assert not x.q.is_cuda and isinstance(x.q, torch.Tensor)


def test_decode_validation_on_host(lib):
    """kda_decode rejects bad arguments before touching CUDA (fake, never-dereferenced pointers)."""
    P = ctypes.c_void_p
    f = [P(0x200000 * (i + 1)) for i in range(7)]
    sc = ctypes.c_float(0.088)

    def call(shape, state=f[5], out=f[6]):
        return lib.kda_decode(ctypes.byref(shape), f[0], f[1], f[2], f[3], f[4], sc, state, out, None)

    ok = _lib.KdaShape(2, 1, 2, 4, 128, 128, 0, _lib.KDA_BF16)
    assert call(ok, state=None) == 1                                               # state is required
    assert call(_lib.KdaShape(1, 1, 2, 4, 128, 128, 1, _lib.KDA_BF16)) == 1         # no packed sequences
    assert call(_lib.KdaShape(2, 1, 3, 4, 128, 128, 0, _lib.KDA_BF16)) == 1         # HV % H != 0
    assert call(_lib.KdaShape(2, 1, 2, 4, 96, 128, 0, _lib.KDA_BF16)) == 2          # K not compiled
    assert call(ok, state=P(0x200000 * 6 + 4)) == 3                                # misaligned state
    assert call(ok, out=f[5]) == 1                                                 # out aliases the state
    assert call(_lib.KdaShape(0, 1, 2, 4, 128, 128, 0, _lib.KDA_BF16)) == 0         # no sequences: nothing to do


def test_gated_validation_on_host(lib):
    """kda_chunk_fwd_gated rejects a missing or malformed gate before touching CUDA."""
    P = ctypes.c_void_p
    f = [P(0x300000 * (i + 1)) for i in range(9)]
    shape = _lib.KdaShape(1, 64, 2, 2, 128, 128, 0, _lib.KDA_BF16)

    def call(gate):
        return lib.kda_chunk_fwd_gated(ctypes.byref(shape), f[0], f[1], f[2], f[3], f[4], gate,
                                       ctypes.c_float(0.088), None, None, f[5], f[6], f[7],
                                       ctypes.c_size_t(1 << 30), None)

    G = _lib.KdaGate
    assert call(None) == 1
    assert call(ctypes.byref(G(0, 0x400000, 0x500000, 0.0))) == 1      # bounded gate needs lower_bound < 0
    assert call(ctypes.byref(G(7, 0x400000, 0x500000, -5.0))) == 1     # unknown gate kind
    assert call(ctypes.byref(G(1, None, 0x500000, 0.0))) == 1          # A_log missing
    assert call(ctypes.byref(G(1, 0x400000, 0x500008, 0.0))) == 3      # dt_bias not 16-byte aligned


def test_backward_validation_on_host(lib):
    """kda_backward sizes its workspace and rejects bad gradients before touching CUDA."""
    P = ctypes.c_void_p
    f = [P(0x10000000 * (i + 1)) for i in range(16)]
    shape = _lib.KdaShape(1, 64, 2, 2, 128, 128, 0, _lib.KDA_BF16)
    need = lib.kda_backward_workspace_size(ctypes.byref(shape))
    assert need == 256 + 2 * (1 + 64) * 128 * 128 * 4            # 1 checkpoint + 64 token states per unit
    sc = ctypes.c_float(0.088)

    def call(ws_bytes=need, **kw):
        a = dict(q=f[0], k=f[1], v=f[2], g=f[3], beta=f[4], s0=None, cu=None, do=f[5], dfin=None,
                 dq=f[6], dk=f[7], dv=f[8], dg=f[9], db=f[10], ds0=f[11], ws=f[12])
        a.update(kw)
        return lib.kda_backward(ctypes.byref(shape), a["q"], a["k"], a["v"], a["g"], a["beta"], sc, a["s0"],
                                a["cu"], a["do"], a["dfin"], a["dq"], a["dk"], a["dv"], a["dg"], a["db"],
                                a["ds0"], a["ws"], ctypes.c_size_t(ws_bytes), None)

    assert call(ws_bytes=need - 1) == 6                    # workspace too small
    assert call(dq=None) == 1                              # gradients are required
    assert call(dq=f[0]) == 1                              # dq aliases q
    assert call(dk=f[6]) == 1                              # dk aliases dq
    assert call(ds0=f[5]) == 1                             # d_initial_state aliases d_out
    assert call(ws=f[2]) == 1                              # the scratch overlaps v
    assert call(dg=P(0x10000000 * 10 + 8)) == 3            # misaligned dg
    assert call(dfin=P(0x10000000 * 14 + 4)) == 3          # misaligned d_final_state
    assert call(do=None) == 1                              # d_out is required
