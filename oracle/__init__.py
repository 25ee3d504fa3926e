"""fp64 CPU oracle for the KDA forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product (the CUDA library and its Python binding)
never imports, links or executes anything under ``oracle/``; the two share no
code.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision), which this
module compiles with gcc and marshals numpy arrays into, and in ``backward_chunked.py``
(plain numpy, double precision).

Forms
-----
``recurrent``: the token recurrence that defines the method
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t
    (the recurrence that ``naive_chunk_kda`` evaluates; page "手撕KDA",
    section "1 Naive").
``chunked``: the chunked WY/UT evaluation in the order of that listing, for
    any chunk size.
``backward``: the gradients of sum <do, o> + <dS_final, S_final> with respect to
    q, k, v, g, beta and the initial state, by reverse mode through the token
    recurrence (the forward re-run with every state kept).
``backward_chunked`` (``backward_chunked.py``, numpy): the same gradients by the chunk
    form of page "手撕KDA", section "2 baseline" (per-chunk recompute, a reverse sweep
    over the states, the VJP of the triangular inverse), every exponential of a
    difference of cumulative decays; a second formulation, pinned against the first.
``prestage`` / ``forward_gated``: the activations applied to raw projections
    before the forward (q/k L2 normalisation with eps 1e-6, the bounded gate
    lower_bound * sigmoid(exp(A_log) (g_raw + dt_bias)) or the softplus gate
    -exp(A_log) softplus(g_raw + dt_bias), beta = sigmoid(beta_raw)); page
    "手撕KDA", sections 2 and 5, and page "KDA源码剖析之FlashKDA（上）", part 7.

Parity status: pinned by the ``-m "not gpu"`` tests in tests/test_oracle_pins.py
(brute-force Kronecker transition, closed forms, textbook delta rule,
hand-computed scalar fixture, invariants).  The pages print no numeric example
for KDA, so no pin is a printed value from the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/_build/libkda_oracle.so with gcc."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.kda_oracle_run.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, P, P, P, P, ctypes.c_double,
                ctypes.c_int, P, P, P, P, P, P, P, P, ctypes.c_int]
            lib.kda_oracle_run.restype = ctypes.c_int
            lib.kda_oracle_tri_inverse.argtypes = [ctypes.c_int, P, P]
            lib.kda_oracle_tri_inverse.restype = None
            lib.kda_oracle_prestage.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                P, P, P, P, P, P, ctypes.c_int, ctypes.c_double, P, P, P, P]
            lib.kda_oracle_prestage.restype = None
            lib.kda_oracle_unit_backward.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, ctypes.c_long, P, ctypes.c_long, P, ctypes.c_long, P, ctypes.c_long, P, ctypes.c_long,
                ctypes.c_double, P, P, P, ctypes.c_long, P, P, P, P, P, P]
            lib.kda_oracle_unit_backward.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def tri_inverse(M: np.ndarray) -> np.ndarray:
    """(I + M)^{-1} for strictly lower-triangular M, by the oracle's forward substitution."""
    M = np.ascontiguousarray(M, dtype=np.float64)
    n = M.shape[0]
    out = np.zeros((n, n), dtype=np.float64)
    _load().kda_oracle_tri_inverse(n, _ptr(M), _ptr(out))
    return out


def _seq_bounds(B, T, cu_seqlens):
    if cu_seqlens is None:
        return [(b * T, T) for b in range(B)]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(int(cu[i]), int(cu[i + 1] - cu[i])) for i in range(len(cu) - 1)]


def forward_units(q, k, v, g, beta, scale, units, initial_state=None, cu_seqlens=None,
                  form: str = "chunked", chunk: int = 64, nthreads: int | None = None):
    """Run the oracle on selected (sequence, value-head) units.

    q, k: [B, T, H, K]; v: [B, T, HV, V]; g: [B, T, HV, K]; beta: [B, T, HV]
    (float32 values; bf16 inputs are passed widened, which is exact).  With
    cu_seqlens ([N+1]) B must be 1 and sequences are packed along T.
    initial_state: [NS, HV, K, V] or None (zeros).
    Returns a list of (o [len, V] float64, S_final [K, V] float64), one per unit.
    """
    q, k, v, g, beta = (_f32(x) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    seqs = _seq_bounds(B, T, cu_seqlens)
    n = len(units)
    tok0 = np.array([seqs[s][0] for s, _ in units], dtype=np.int64)
    lens = np.array([seqs[s][1] for s, _ in units], dtype=np.int32)
    hvs = np.array([h for _, h in units], dtype=np.int32)
    o_off = np.zeros(n, dtype=np.int64)
    if n:
        o_off[1:] = np.cumsum(lens.astype(np.int64) * V)[:-1]
    o_out = np.zeros(int(lens.astype(np.int64).sum()) * V, dtype=np.float64)
    s_out = np.zeros((n, K, V), dtype=np.float64)
    s0 = None
    s0_off = None
    if initial_state is not None:
        s0 = _f32(initial_state)
        s0_off = np.array([(s * HV + h) * K * V for s, h in units], dtype=np.int64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().kda_oracle_run(
        0 if form == "recurrent" else 1, int(chunk), H, HV, K, V,
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        n, _ptr(tok0), _ptr(lens), _ptr(hvs), _ptr(s0), _ptr(s0_off),
        _ptr(o_out), _ptr(o_off), _ptr(s_out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    res = []
    for i in range(n):
        L = int(lens[i])
        res.append((o_out[o_off[i]:o_off[i] + L * V].reshape(L, V), s_out[i]))
    return res


def forward(q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None,
            form: str = "chunked", chunk: int = 64, nthreads: int | None = None):
    """Run the oracle on every unit.  Returns (o [B,T,HV,V] f64, S [NS,HV,K,V] f64)."""
    B, T = np.shape(q)[0], np.shape(q)[1]
    HV, V = np.shape(v)[2], np.shape(v)[3]
    K = np.shape(q)[3]
    seqs = _seq_bounds(B, T, cu_seqlens)
    units = [(s, h) for s in range(len(seqs)) for h in range(HV)]
    res = forward_units(q, k, v, g, beta, scale, units, initial_state, cu_seqlens,
                        form, chunk, nthreads)
    o = np.zeros((B * T, HV, V), dtype=np.float64)
    S = np.zeros((len(seqs), HV, K, V), dtype=np.float64)
    for (s, h), (ou, su) in zip(units, res):
        t0, L = seqs[s]
        o[t0:t0 + L, h, :] = ou
        S[s, h] = su
    return o.reshape(B, T, HV, V), S


GATES = {"bounded": 0, "softplus": 1}


def prestage(q_raw, k_raw, g_raw, beta_raw, A_log, dt_bias, gate: str = "bounded", lower_bound: float = -5.0):
    """The forward's inputs from raw projections, in fp64 (see kda_oracle_prestage).
    q_raw, k_raw [B, T, H, K]; g_raw [B, T, HV, K]; beta_raw [B, T, HV]; A_log [HV];
    dt_bias [HV, K].  Returns (q, k, g, beta) as float64 arrays of the same shapes."""
    q_raw, k_raw, g_raw, beta_raw, A_log, dt_bias = (_f32(x) for x in (q_raw, k_raw, g_raw, beta_raw, A_log, dt_bias))
    B, T, H, K = q_raw.shape
    HV = g_raw.shape[2]
    n = B * T
    q = np.zeros(q_raw.shape, dtype=np.float64)
    k = np.zeros(k_raw.shape, dtype=np.float64)
    g = np.zeros(g_raw.shape, dtype=np.float64)
    beta = np.zeros(beta_raw.shape, dtype=np.float64)
    _load().kda_oracle_prestage(n, H, HV, K, _ptr(q_raw), _ptr(k_raw), _ptr(g_raw), _ptr(beta_raw), _ptr(A_log),
                                _ptr(dt_bias), GATES[gate], float(lower_bound), _ptr(q), _ptr(k), _ptr(g), _ptr(beta))
    return q, k, g, beta


def forward_gated(q_raw, k_raw, v, g_raw, beta_raw, A_log, dt_bias, scale, gate: str = "bounded",
                  lower_bound: float = -5.0, initial_state=None, cu_seqlens=None, form: str = "recurrent",
                  chunk: int = 64, nthreads: int | None = None):
    """prestage() then forward().  The pre-stage is evaluated in fp64; forward() reads
    its results rounded to fp32 (a relative change of at most 6e-8, far below any
    tolerance this oracle is used with)."""
    q, k, g, beta = prestage(q_raw, k_raw, g_raw, beta_raw, A_log, dt_bias, gate, lower_bound)
    return forward(q, k, v, g, beta, scale, initial_state=initial_state, cu_seqlens=cu_seqlens, form=form,
                   chunk=chunk, nthreads=nthreads)


def backward(q, k, v, g, beta, scale, do, d_final_state=None, initial_state=None, cu_seqlens=None):
    """Gradients of sum_t <do_t, o_t> + <d_final_state, S_final> (see kda_oracle_unit_backward).
    Shapes as forward(); do [B, T, HV, V]; d_final_state [NS, HV, K, V] or None.  dq and dk
    of a key head sum the contributions of the value heads that share it.  Returns
    (dq [B,T,H,K], dk [B,T,H,K], dv [B,T,HV,V], dg [B,T,HV,K], dbeta [B,T,HV],
    d_initial_state [NS,HV,K,V]), all float64."""
    q, k, v, g, beta, do = (_f32(x) for x in (q, k, v, g, beta, do))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    seqs = _seq_bounds(B, T, cu_seqlens)
    qf, kf, vf, gf, bf, dof = (a.reshape((B * T,) + a.shape[2:]) for a in (q, k, v, g, beta, do))
    dq = np.zeros((B * T, H, K))
    dk = np.zeros((B * T, H, K))
    dv = np.zeros((B * T, HV, V))
    dg = np.zeros((B * T, HV, K))
    db = np.zeros((B * T, HV))
    ds0 = np.zeros((len(seqs), HV, K, V))
    lib = _load()
    for s, (t0, L) in enumerate(seqs):
        for h in range(HV):
            hk = h // G
            s0 = None if initial_state is None else np.ascontiguousarray(np.asarray(initial_state)[s, h], dtype=np.float64)
            dfin = None if d_final_state is None else np.ascontiguousarray(np.asarray(d_final_state)[s, h], dtype=np.float64)
            do_u = np.ascontiguousarray(dof[t0:t0 + L, h], dtype=np.float64)
            dq_u, dk_u, dv_u = np.zeros((L, K)), np.zeros((L, K)), np.zeros((L, V))
            dg_u, db_u, ds_u = np.zeros((L, K)), np.zeros(L), np.zeros((K, V))
            if L:
                lib.kda_oracle_unit_backward(
                    L, K, V, _ptr(np.ascontiguousarray(qf[t0:t0 + L, hk])), K, _ptr(np.ascontiguousarray(kf[t0:t0 + L, hk])), K,
                    _ptr(np.ascontiguousarray(vf[t0:t0 + L, h])), V, _ptr(np.ascontiguousarray(gf[t0:t0 + L, h])), K,
                    _ptr(np.ascontiguousarray(bf[t0:t0 + L, h])), 1, float(scale), _ptr(s0), _ptr(dfin), _ptr(do_u), V,
                    _ptr(dq_u), _ptr(dk_u), _ptr(dv_u), _ptr(dg_u), _ptr(db_u), _ptr(ds_u))
            else:
                ds_u = np.zeros((K, V)) if dfin is None else dfin.copy()
            dq[t0:t0 + L, hk] += dq_u
            dk[t0:t0 + L, hk] += dk_u
            dv[t0:t0 + L, h] = dv_u
            dg[t0:t0 + L, h] = dg_u
            db[t0:t0 + L, h] = db_u
            ds0[s, h] = ds_u
    r = lambda a: a.reshape((B, T) + a.shape[1:])
    return r(dq), r(dk), r(dv), r(dg), r(db), ds0


from .backward_chunked import backward_chunked  # noqa: E402  (the chunk-form backward)
