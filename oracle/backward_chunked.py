"""fp64 chunk-form backward of KDA -- TEST INFRASTRUCTURE ONLY (part of ``oracle``).

A second, independent formulation of the gradients that ``oracle.backward`` takes by
reverse mode through the token recurrence: the steps of the chunked backward of page
"手撕KDA", section "2 baseline" (2.1, the C++ port: the forward re-run chunk by chunk
keeping the state entering each chunk, then a sweep over the chunks in reverse carrying
the state's gradient, with the VJP of the chunk's triangular inverse), written in plain
numpy in double precision from the chain rule through the chunked form of section
"1 Naive".  Every exponential is taken of a difference of cumulative decays, as the
oracle's forward does, so no factor overflows for strong gates.

Notation per chunk (rows i, j; gc the cumulative sum of g from the chunk start, gl its
last row, S the state entering the chunk):
    M_ij = beta_i sum_d k_id k_jd e^{gc_id - gc_jd}   (j < i),   T = (I + M)^{-1},  A = T Diag(beta)
    Aqk_ij = scale sum_d q_id k_jd e^{gc_id - gc_jd}  (j <= i)
    W = A (k e^{gc}),  U = A v,  v_new = U - W S
    o = (scale q e^{gc}) S + Aqk v_new,   S' = Diag(e^{gl}) S + (k e^{gl - gc})^T v_new
"""
from __future__ import annotations

import numpy as np


def _decay(gc: np.ndarray) -> np.ndarray:
    """e^{gc_i - gc_j} per key dim for j <= i, zero above the diagonal: [C, C, K] (row i,
    column j).  Every exponent taken is <= 0."""
    c = gc.shape[0]
    diff = gc[:, None, :] - gc[None, :, :]
    lower = np.tril(np.ones((c, c), dtype=bool))[:, :, None]
    return np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)


def _unit(q, k, v, g, beta, scale, do, s0, dfin, C):
    """Gradients of one (sequence, value head) unit; q, k of its key head.  Returns
    (dq, dk, dv, dg, dbeta, d_initial_state)."""
    L, K = q.shape
    V = v.shape[1]
    chunks = [(c0, min(C, L - c0)) for c0 in range(0, L, C)]
    # forward, keeping the state entering every chunk
    S = np.zeros((K, V)) if s0 is None else s0.copy()
    entering = []
    for c0, c in chunks:
        entering.append(S.copy())
        sl = slice(c0, c0 + c)
        gc = np.cumsum(g[sl], axis=0)
        gl = gc[-1]
        E = _decay(gc)
        kk, bb = k[sl], beta[sl]
        M = np.tril(bb[:, None] * np.einsum("id,jd,ijd->ij", kk, kk, E), -1)
        T = np.linalg.solve(np.eye(c) + M, np.eye(c))
        A = T * bb[None, :]
        W = A @ (kk * np.exp(gc))
        v_new = A @ v[sl] - W @ S
        S = np.exp(gl)[:, None] * S + (kk * np.exp(gl - gc)).T @ v_new
    # the reverse sweep
    dq, dk, dv, dg, db = (np.zeros_like(a) for a in (q, k, v, g, beta))
    dS = np.zeros((K, V)) if dfin is None else dfin.copy()  # the gradient of the state leaving the chunk
    for n in range(len(chunks) - 1, -1, -1):
        c0, c = chunks[n]
        sl = slice(c0, c0 + c)
        h = entering[n]
        qq, kk, vv, bb, dd = q[sl], k[sl], v[sl], beta[sl], do[sl]
        gc = np.cumsum(g[sl], axis=0)
        gl = gc[-1]
        E = _decay(gc)
        low = np.tril(np.ones((c, c)))              # j <= i
        strict = np.tril(np.ones((c, c)), -1)       # j < i
        KK = np.einsum("id,jd,ijd->ij", kk, kk, E) * strict
        M = bb[:, None] * KK
        T = np.linalg.solve(np.eye(c) + M, np.eye(c))
        A = T * bb[None, :]
        kd = kk * np.exp(gc)
        kr = kk * np.exp(gl - gc)
        qd = scale * qq * np.exp(gc)
        Aqk = scale * np.einsum("id,jd,ijd->ij", qq, kk, E) * low
        W = A @ kd
        v_new = A @ vv - W @ h
        # o = qd h + Aqk v_new;  S' = e^{gl} h + kr^T v_new
        d_vnew = Aqk.T @ dd + kr @ dS
        d_Aqk = (dd @ v_new.T) * low
        d_h = qd.T @ dd + np.exp(gl)[:, None] * dS
        d_qd = dd @ h.T
        d_kr = v_new @ dS.T
        d_gl = np.exp(gl) * np.sum(h * dS, axis=1)
        # v_new = U - W h, U = A v, W = A kd
        d_W = -d_vnew @ h.T
        d_h -= W.T @ d_vnew
        d_A = d_W @ kd.T + d_vnew @ vv.T
        d_kd = A.T @ d_W
        dv[sl] = A.T @ d_vnew
        # A = T Diag(beta), T = (I + M)^{-1}, M = Diag(beta) KK (strictly lower)
        d_T = d_A * bb[None, :]
        d_beta = np.sum(T * d_A, axis=0)
        d_M = -(T.T @ d_T @ T.T) * strict
        d_beta += np.sum(d_M * KK, axis=1)
        d_KK = bb[:, None] * d_M
        # the decayed products: KK_ij = sum_d k_id k_jd e^{gc_id - gc_jd} (j < i),
        # Aqk_ij = scale sum_d q_id k_jd e^{gc_id - gc_jd} (j <= i)
        d_q = scale * np.einsum("ij,jd,ijd->id", d_Aqk, kk, E)
        d_k = np.einsum("ij,jd,ijd->id", d_KK, kk, E) + np.einsum("ij,id,ijd->jd", d_KK, kk, E) \
            + scale * np.einsum("ij,id,ijd->jd", d_Aqk, qq, E)
        # d/d gc of those products: + on the row side (i), - on the column side (j)
        d_gc = kk * np.einsum("ij,jd,ijd->id", d_KK, kk, E) - kk * np.einsum("ij,id,ijd->jd", d_KK, kk, E) \
            + qq * d_q - kk * scale * np.einsum("ij,id,ijd->jd", d_Aqk, qq, E)
        # kd = k e^{gc}, qd = scale q e^{gc}, kr = k e^{gl - gc}
        d_k += d_kd * np.exp(gc) + d_kr * np.exp(gl - gc)
        d_q += scale * d_qd * np.exp(gc)
        d_gc += d_kd * kd + d_qd * qd - d_kr * kr
        d_gl += np.sum(d_kr * kr, axis=0)
        d_gc[-1] += d_gl
        dq[sl], dk[sl], db[sl] = d_q, d_k, d_beta
        dg[sl] = np.cumsum(d_gc[::-1], axis=0)[::-1]  # gc = cumsum(g)
        dS = d_h
    return dq, dk, dv, dg, db, dS


def backward_chunked(q, k, v, g, beta, scale, do, d_final_state=None, initial_state=None, cu_seqlens=None,
                     chunk: int = 64):
    """The same gradients as ``oracle.backward`` (same shapes and conventions: dq and dk of
    a key head sum its value heads), by the chunk form above with chunks of ``chunk``
    tokens.  All float64."""
    f = lambda a: None if a is None else np.asarray(a, dtype=np.float64)
    q, k, v, g, beta, do = (f(a) for a in (q, k, v, g, beta, do))
    s0, dfin = f(initial_state), f(d_final_state)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        seqs = [(0, int(cu[i]), int(cu[i + 1] - cu[i])) for i in range(len(cu) - 1)]
    dq, dk = np.zeros((B, T, H, K)), np.zeros((B, T, H, K))
    dv, dg, db = np.zeros((B, T, HV, V)), np.zeros((B, T, HV, K)), np.zeros((B, T, HV))
    ds0 = np.zeros((len(seqs), HV, K, V))
    for s, (b, t0, L) in enumerate(seqs):
        ts = slice(t0, t0 + L)
        for hv in range(HV):
            hk = hv // G
            si = None if s0 is None else s0[s, hv]
            di = None if dfin is None else dfin[s, hv]
            if L == 0:
                ds0[s, hv] = np.zeros((K, V)) if di is None else di
                continue
            r = _unit(q[b, ts, hk], k[b, ts, hk], v[b, ts, hv], g[b, ts, hv], beta[b, ts, hv], scale, do[b, ts, hv],
                      si, di, chunk)
            dq[b, ts, hk] += r[0]
            dk[b, ts, hk] += r[1]
            dv[b, ts, hv], dg[b, ts, hv], db[b, ts, hv], ds0[s, hv] = r[2], r[3], r[4], r[5]
    return dq, dk, dv, dg, db, ds0
