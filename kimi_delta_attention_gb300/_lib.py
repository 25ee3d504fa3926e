"""ctypes binding of the C ABI in include/kda.h (argument marshalling only).

Every step of the forward runs in the CUDA library libkda.so; this module only
turns torch tensors into device pointers and sizes, allocates outputs with
torch when the caller did not pass them, and raises on a non-OK status.  There
is no fallback: if the library is missing the call fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import builder as _build

_lock = threading.Lock()
_lib = None

KDA_F32 = 0
KDA_BF16 = 1

STATUS_NAMES = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_ALIGNMENT",
    4: "KDA_ERR_CUDA", 5: "KDA_ERR_DEVICE_TIMEOUT", 6: "KDA_ERR_WORKSPACE", 7: "KDA_ERR_DEVICE_BOUNDS",
    8: "KDA_ERR_STATIC_SCRATCH", 9: "KDA_ERR_DECAY_RANGE",
}
STATIC_SCRATCH_MAX_UNITS = 32

# Every symbol include/kda.h declares.
EXPORTS = ("kda_chunk_fwd", "kda_recurrent_fwd", "kda_chunk_fwd_workspace_size",
           "kda_read_device_status", "kda_status_string", "kda_chunk_size",
           "kda_chunk_fwd_kernel_name", "kda_chunk_fwd_kernel_launches", "kda_chunk_fwd_static_scratch", "kda_decode", "kda_chunk_fwd_gated",
           "kda_chunk_states_size", "kda_chunk_states", "kda_chunk_output", "kda_backward_workspace_size",
           "kda_backward")
GATE_KINDS = {"bounded": 0, "softplus": 1}


class KdaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class KdaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("HV", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("io_dtype", ctypes.c_int)]


class KdaGate(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("lower_bound", ctypes.c_float)]


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libkda.so (built in-tree by kimi_delta_attention_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"KDA CUDA library not built ({p}); run kimi_delta_attention_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        fwd_args = [ctypes.POINTER(KdaShape), P, P, P, P, P, F, P, P, P, P, P, S, P]
        for name in ("kda_chunk_fwd", "kda_recurrent_fwd"):
            fn = getattr(lib, name)
            fn.argtypes = fwd_args
            fn.restype = I
        lib.kda_chunk_fwd_workspace_size.argtypes = [ctypes.POINTER(KdaShape)]
        lib.kda_chunk_fwd_workspace_size.restype = S
        lib.kda_read_device_status.argtypes = [P, P]
        lib.kda_read_device_status.restype = I
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_chunk_size.argtypes = []
        lib.kda_chunk_size.restype = I
        lib.kda_chunk_fwd_kernel_name.argtypes = [ctypes.POINTER(KdaShape)]
        lib.kda_chunk_fwd_kernel_name.restype = ctypes.c_char_p
        lib.kda_chunk_fwd_kernel_launches.argtypes = [ctypes.POINTER(KdaShape)]
        lib.kda_chunk_fwd_kernel_launches.restype = I
        lib.kda_chunk_fwd_static_scratch.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, F, P, P, P, P, P,
                                                     ctypes.POINTER(ctypes.c_void_p)]
        lib.kda_chunk_fwd_static_scratch.restype = I
        lib.kda_decode.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, F, P, P, P]
        lib.kda_decode.restype = I
        lib.kda_chunk_fwd_gated.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, ctypes.POINTER(KdaGate), F,
                                            P, P, P, P, P, S, P]
        lib.kda_chunk_fwd_gated.restype = I
        lib.kda_chunk_states_size.argtypes = [ctypes.POINTER(KdaShape)]
        lib.kda_chunk_states_size.restype = S
        lib.kda_chunk_states.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, P, P, P, P, S, P]
        lib.kda_chunk_states.restype = I
        lib.kda_chunk_output.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, F, P, P, P, S, P]
        lib.kda_chunk_output.restype = I
        lib.kda_backward_workspace_size.argtypes = [ctypes.POINTER(KdaShape)]
        lib.kda_backward_workspace_size.restype = S
        lib.kda_backward.argtypes = [ctypes.POINTER(KdaShape), P, P, P, P, P, F, P, P, P, P,
                                     P, P, P, P, P, P, P, S, P]
        lib.kda_backward.restype = I
        if path is None:
            _lib = lib
        return lib


def kda_status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def _check(code: int):
    if code != 0:
        raise KdaError(code, kda_status_string(code))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_shape(q, v, cu_seqlens=None) -> KdaShape:
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    io = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}.get(q.dtype)
    if io is None:
        raise KdaError(1, f"unsupported io dtype {q.dtype}")
    ns = 0 if cu_seqlens is None else int(cu_seqlens.numel()) - 1
    return KdaShape(B, T, H, HV, K, V, ns, io)


def kda_chunk_fwd_workspace_size(shape: KdaShape) -> int:
    return int(load_library().kda_chunk_fwd_workspace_size(ctypes.byref(shape)))


def kda_chunk_size() -> int:
    return int(load_library().kda_chunk_size())


def kda_chunk_fwd_kernel_name(shape: KdaShape) -> str:
    """Kernel kda_chunk_fwd launches for `shape` on the current device."""
    return load_library().kda_chunk_fwd_kernel_name(ctypes.byref(shape)).decode()


def kda_chunk_fwd_kernel_launches(shape: KdaShape) -> int:
    """How many launches of that kernel one kda_chunk_fwd call makes."""
    return int(load_library().kda_chunk_fwd_kernel_launches(ctypes.byref(shape)))


def _check_tensors(q, k, v, g, beta, others):
    """Inputs must be contiguous CUDA tensors; every tensor handed to the library must
    live on q's device (the call runs with that device current)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise KdaError(1, f"{name} must be a contiguous CUDA tensor")
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta)) + tuple(others):
        if t is not None and t.device != q.device:
            raise KdaError(1, f"{name} is on {t.device}, q on {q.device}")


def _forward(entry: str, q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
             out=None, final_state=None, output_final_state=True, workspace=None, stream=None):
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("initial_state", initial_state), ("cu_seqlens", cu_seqlens),
                                      ("out", out), ("final_state", final_state), ("workspace", workspace)))
    with torch.cuda.device(q.device):
        return _forward_on_device(lib, entry, q, k, v, g, beta, scale, initial_state, cu_seqlens, out,
                                  final_state, output_final_state, workspace, stream)


def _forward_on_device(lib, entry, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state,
                       output_final_state, workspace, stream):
    shape = make_shape(q, v, cu_seqlens)
    K = q.shape[3]
    if scale is None:
        scale = K ** -0.5
    NS = q.shape[0] if cu_seqlens is None else shape.num_seqs
    HV, V = v.shape[2], v.shape[3]
    made = []  # tensors allocated here, on the current stream's pool
    if out is None:
        out = torch.empty_like(v)
        made.append(out)
    if final_state is None and output_final_state:
        final_state = torch.empty((NS, HV, K, V), dtype=torch.float32, device=q.device)
        made.append(final_state)
    if workspace is None:
        workspace = torch.empty(kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device=q.device)
        made.append(workspace)
    current = torch.cuda.current_stream(q.device).cuda_stream
    if stream is None:
        stream = current
    code = getattr(lib, entry)(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), ctypes.c_void_p(stream))
    _check(code)
    if made and stream != current:
        # the work runs on another stream: the caching allocator must not hand these blocks
        # (the temporary workspace above all) to the current stream before that work is done
        other = torch.cuda.ExternalStream(stream, device=q.device)
        for t in made:
            t.record_stream(other)
    return out, final_state


def kda_chunk_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None, out=None,
                  final_state=None, output_final_state=True, workspace=None, stream=None):
    """Chunked KDA forward on the GPU.  Shapes: q, k [B,T,H,K]; v [B,T,HV,V];
    g [B,T,HV,K] fp32; beta [B,T,HV] fp32; initial_state [NS,HV,K,V] fp32;
    cu_seqlens [N+1] int32.  Returns (o [B,T,HV,V], final_state or None)."""
    return _forward("kda_chunk_fwd", q, k, v, g, beta, scale, initial_state, cu_seqlens, out,
                    final_state, output_final_state, workspace, stream)


def kda_recurrent_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None, out=None,
                      final_state=None, output_final_state=True, workspace=None, stream=None):
    """Token-recurrent KDA forward on the GPU (same arguments and results)."""
    return _forward("kda_recurrent_fwd", q, k, v, g, beta, scale, initial_state, cu_seqlens, out,
                    final_state, output_final_state, workspace, stream)


def kda_read_device_status(workspace, stream=None) -> int:
    with torch.cuda.device(workspace.device):
        if stream is None:
            stream = torch.cuda.current_stream(workspace.device).cuda_stream
        return int(load_library().kda_read_device_status(_ptr(workspace), ctypes.c_void_p(stream)))


def kda_chunk_fwd_static_scratch(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                                 out=None, final_state=None, output_final_state=True, stream=None):
    """kda_chunk_fwd for callers that cannot hand over device scratch: the library's
    fixed array holds it (at most 32 (sequence, value head) pairs per call; calls
    that overlap on the GPU race).  Returns (o, final_state, status_word_address)."""
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("initial_state", initial_state), ("cu_seqlens", cu_seqlens),
                                      ("out", out), ("final_state", final_state)))
    with torch.cuda.device(q.device):
        shape = make_shape(q, v, cu_seqlens)
        K = q.shape[3]
        if scale is None:
            scale = K ** -0.5
        NS = q.shape[0] if cu_seqlens is None else shape.num_seqs
        HV, V = v.shape[2], v.shape[3]
        if out is None:
            out = torch.empty_like(v)
        if final_state is None and output_final_state:
            final_state = torch.empty((NS, HV, K, V), dtype=torch.float32, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device).cuda_stream
        status = ctypes.c_void_p()
        code = lib.kda_chunk_fwd_static_scratch(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
            _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state), ctypes.c_void_p(stream),
            ctypes.byref(status))
        _check(code)
    return out, final_state, status.value


def kda_decode(q, k, v, g, beta, state, scale=None, out=None, stream=None):
    """Recurrent step for inference: q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV,K] fp32;
    beta [B,T,HV] fp32; state [B,HV,K,V] fp32, updated in place.  Returns o [B,T,HV,V]."""
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("state", state), ("out", out)))
    if state is None or not state.is_contiguous() or state.dtype != torch.float32:
        raise KdaError(1, "state must be a contiguous fp32 CUDA tensor")
    with torch.cuda.device(q.device):
        shape = make_shape(q, v)
        if scale is None:
            scale = q.shape[3] ** -0.5
        if out is None:
            out = torch.empty_like(v)
        if stream is None:
            stream = torch.cuda.current_stream(q.device).cuda_stream
        _check(lib.kda_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              ctypes.c_float(scale), _ptr(state), _ptr(out), ctypes.c_void_p(stream)))
    return out


def kda_chunk_fwd_gated(q, k, v, g_raw, beta_raw, A_log, dt_bias, gate="bounded", lower_bound=-5.0, scale=None,
                        initial_state=None, cu_seqlens=None, out=None, final_state=None, output_final_state=True,
                        workspace=None, stream=None):
    """Chunked forward with the pre-stage fused in: raw q, k [B,T,H,K] bf16 (L2-normalised
    in the kernel), v [B,T,HV,V] bf16, g_raw [B,T,HV,K] bf16, beta_raw [B,T,HV] fp32,
    A_log [HV] and dt_bias [HV,K] fp32; gate "bounded" (lower_bound sigmoid(exp(A_log)
    (g_raw + dt_bias))) or "softplus" (-exp(A_log) softplus(g_raw + dt_bias))."""
    lib = load_library()
    _check_tensors(q, k, v, g_raw, beta_raw, (("A_log", A_log), ("dt_bias", dt_bias),
                                              ("initial_state", initial_state), ("cu_seqlens", cu_seqlens),
                                              ("out", out), ("final_state", final_state), ("workspace", workspace)))
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise KdaError(1, f"{name} must be a contiguous fp32 CUDA tensor")
    with torch.cuda.device(q.device):
        shape = make_shape(q, v, cu_seqlens)
        K = q.shape[3]
        if scale is None:
            scale = K ** -0.5
        NS = q.shape[0] if cu_seqlens is None else shape.num_seqs
        HV, V = v.shape[2], v.shape[3]
        made = []
        if out is None:
            out = torch.empty_like(v)
            made.append(out)
        if final_state is None and output_final_state:
            final_state = torch.empty((NS, HV, K, V), dtype=torch.float32, device=q.device)
            made.append(final_state)
        if workspace is None:
            workspace = torch.empty(kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device=q.device)
            made.append(workspace)
        current = torch.cuda.current_stream(q.device).cuda_stream
        if stream is None:
            stream = current
        gs = KdaGate(GATE_KINDS[gate], A_log.data_ptr(), dt_bias.data_ptr(), float(lower_bound))
        _check(lib.kda_chunk_fwd_gated(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw), ctypes.byref(gs),
            ctypes.c_float(scale), _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
            _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()), ctypes.c_void_p(stream)))
        if made and stream != current:
            other = torch.cuda.ExternalStream(stream, device=q.device)
            for t in made:
                t.record_stream(other)
    return out, final_state


def kda_chunk_states(q, k, v, g, beta, initial_state=None, h=None, final_state=None, output_final_state=True,
                     workspace=None, stream=None):
    """The state scan alone: h [B, HV, NT, K, V] bf16 (the state entering each chunk of 64
    tokens) and the final state.  Fixed-length bf16, K = V = 128.  Returns (h, final_state)."""
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("initial_state", initial_state), ("h", h), ("final_state", final_state),
                                      ("workspace", workspace)))
    with torch.cuda.device(q.device):
        shape = make_shape(q, v)
        B, T, H, K = q.shape
        HV, V = v.shape[2], v.shape[3]
        if h is None:
            h = torch.empty((B, HV, (T + 63) // 64, K, V), dtype=torch.bfloat16, device=q.device)
        if final_state is None and output_final_state:
            final_state = torch.empty((B, HV, K, V), dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = torch.empty(kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device).cuda_stream
        _check(lib.kda_chunk_states(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(initial_state), _ptr(h), _ptr(final_state), _ptr(workspace),
                                    ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                    ctypes.c_void_p(stream)))
    return h, final_state


def kda_chunk_output(q, k, v, g, beta, h, scale=None, out=None, workspace=None, stream=None):
    """o of every chunk in parallel from the states h (as kda_chunk_states writes them)."""
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("h", h), ("out", out), ("workspace", workspace)))
    with torch.cuda.device(q.device):
        shape = make_shape(q, v)
        if scale is None:
            scale = q.shape[3] ** -0.5
        if out is None:
            out = torch.empty_like(v)
        if workspace is None:
            workspace = torch.empty(256, dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device).cuda_stream
        _check(lib.kda_chunk_output(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    ctypes.c_float(scale), _ptr(h), _ptr(out), _ptr(workspace),
                                    ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                    ctypes.c_void_p(stream)))
    return out


def kda_backward_workspace_size(shape: KdaShape) -> int:
    return int(load_library().kda_backward_workspace_size(ctypes.byref(shape)))


def kda_backward(q, k, v, g, beta, d_out, scale=None, initial_state=None, cu_seqlens=None, d_final_state=None,
                 output_d_initial_state=True, workspace=None, stream=None):
    """Gradients of sum <d_out, o> + <d_final_state, S_final> for the forward with the same
    arguments.  d_out [B,T,HV,V] in q's dtype, d_final_state [NS,HV,K,V] fp32 or None.
    Returns (dq, dk, dv, dg, dbeta, d_initial_state), all fp32, in the inputs' shapes."""
    lib = load_library()
    _check_tensors(q, k, v, g, beta, (("d_out", d_out), ("initial_state", initial_state),
                                      ("cu_seqlens", cu_seqlens), ("d_final_state", d_final_state),
                                      ("workspace", workspace)))
    if not d_out.is_contiguous() or d_out.dtype != q.dtype:
        raise KdaError(1, "d_out must be contiguous with q's dtype")
    with torch.cuda.device(q.device):
        shape = make_shape(q, v, cu_seqlens)
        K = q.shape[3]
        if scale is None:
            scale = K ** -0.5
        NS = q.shape[0] if cu_seqlens is None else shape.num_seqs
        HV, V = v.shape[2], v.shape[3]
        f32 = dict(dtype=torch.float32, device=q.device)
        dq = torch.empty(q.shape, **f32)
        dk = torch.empty(k.shape, **f32)
        dv = torch.empty(v.shape, **f32)
        dg = torch.empty(g.shape, **f32)
        dbeta = torch.empty(beta.shape, **f32)
        ds0 = torch.empty((NS, HV, K, V), **f32) if output_d_initial_state else None
        made = [dq, dk, dv, dg, dbeta] + ([ds0] if ds0 is not None else [])
        if workspace is None:
            workspace = torch.empty(kda_backward_workspace_size(shape), dtype=torch.uint8, device=q.device)
            made.append(workspace)
        current = torch.cuda.current_stream(q.device).cuda_stream
        if stream is None:
            stream = current
        _check(lib.kda_backward(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), ctypes.c_float(scale),
            _ptr(initial_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(dg), _ptr(dbeta), _ptr(ds0), _ptr(workspace),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), ctypes.c_void_p(stream)))
        if stream != current:
            other = torch.cuda.ExternalStream(stream, device=q.device)
            for t in made:
                t.record_stream(other)
    return dq, dk, dv, dg, dbeta, ds0
