"""Shared helpers for the GPU parity tests: run the oracle on the exact inputs
handed to the GPU and compare with the tolerances the method's statement fixes."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances (from the statement of the forward's accuracy bar):
#   bf16 I/O: max|o - o_ref| <= 2e-2 * max|o_ref|, ||S - S_ref||_F <= 1e-2 ||S_ref||_F
#   fp32 I/O: ||S - S_ref||_F <= 1e-4 ||S_ref||_F; o is held to the same 1e-4 (of max|o_ref|),
#   which the fp32 token recurrence meets with a wide margin (errors ~1e-6).
TOL = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 1e-4)}


def np32(t):
    return None if t is None else t.detach().to("cpu", torch.float32).numpy()


def oracle_full(x, form="recurrent", chunk=64):
    return oracle.forward(np32(x.q), np32(x.k), np32(x.v), np32(x.g), np32(x.beta), x.scale,
                          initial_state=np32(x.initial_state),
                          cu_seqlens=None if x.cu_seqlens is None else x.cu_seqlens.numpy(),
                          form=form, chunk=chunk)


def oracle_units(x, units, form="recurrent", chunk=64):
    return oracle.forward_units(np32(x.q), np32(x.k), np32(x.v), np32(x.g), np32(x.beta), x.scale, units,
                                initial_state=np32(x.initial_state),
                                cu_seqlens=None if x.cu_seqlens is None else x.cu_seqlens.numpy(),
                                form=form, chunk=chunk)


def seq_bounds(x):
    if x.cu_seqlens is None:
        T = x.q.shape[1]
        return [(b * T, T) for b in range(x.q.shape[0])]
    cu = x.cu_seqlens.numpy().astype(np.int64)
    return [(int(cu[i]), int(cu[i + 1] - cu[i])) for i in range(len(cu) - 1)]


def errors(o, S, o_ref, S_ref):
    """(max|o - o_ref| / max|o_ref|, ||S - S_ref||_F / ||S_ref||_F)."""
    o = np.asarray(o, dtype=np.float64)
    eo = np.abs(o - o_ref).max() / max(np.abs(o_ref).max(), 1e-30) if o_ref.size else 0.0
    es = 0.0
    if S is not None:
        S = np.asarray(S, dtype=np.float64)
        es = np.linalg.norm(S - S_ref) / max(np.linalg.norm(S_ref), 1e-30)
    return eo, es


def assert_close(o, S, o_ref, S_ref, io, what=""):
    to, ts = TOL[io]
    eo, es = errors(o, S, o_ref, S_ref)
    assert np.all(np.isfinite(np.asarray(o))), f"{what}: non-finite output"
    assert eo <= to, f"{what}: o error {eo:.3e} > {to}"
    assert es <= ts, f"{what}: state error {es:.3e} > {ts}"
    return eo, es


def check_units(x, o_gpu, S_gpu, units, form="recurrent"):
    """Compare the GPU result on selected (sequence, value head) units."""
    res = oracle_units(x, units, form=form)
    bounds = seq_bounds(x)
    HV, V = x.v.shape[2], x.v.shape[3]
    o_flat = o_gpu.reshape(-1, HV, V)
    worst = (0.0, 0.0)
    for (s, h), (o_ref, S_ref) in zip(units, res):
        t0, L = bounds[s]
        o_u = o_flat[t0:t0 + L, h, :].float().cpu().numpy()
        S_u = None if S_gpu is None else S_gpu[s, h].float().cpu().numpy()
        e = assert_close(o_u, S_u, o_ref, S_ref if S_gpu is not None else None, x.io_dtype,
                         what=f"unit {(s, h)}")
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    return worst


def check_all_units(x, o_gpu, S_gpu, block=64, form="recurrent"):
    """Compare the GPU result with the oracle on every (sequence, value head) unit,
    `block` units per oracle call (the oracle runs them on all host cores)."""
    HV = x.v.shape[2]
    units = [(s, h) for s in range(x.num_seqs) for h in range(HV)]
    worst = (0.0, 0.0)
    for i in range(0, len(units), block):
        e = check_units(x, o_gpu, S_gpu, units[i:i + block], form=form)
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    return worst
