"""Seeded synthetic inputs for the KDA chunked forward.

This module holds the input recipe only -- none of the method's arithmetic.
Both the CUDA path (tests, benchmark) and the fp64 oracle consume the tensors
made here; the oracle reads the exact bytes handed to the GPU, widened to fp32.

Recipe (the same for every workload):
  * numpy PCG64 generator seeded with the workload index; draw order:
    sequence lengths (varlen only), q, k, v, g, beta, initial state.
  * q, k ~ N(0, 1) per element, then divided by their L2 norm per (token, head)
    in fp32 (plain x / ||x||), then cast to the I/O dtype.
  * v ~ N(0, 1), cast to the I/O dtype.
  * g = logsigmoid(N(0, 1)) / 8 per (token, value head, key dim): a log-space
    decay <= 0, kept in fp32.
  * beta = sigmoid(N(0, 1)) per (token, value head), fp32.
  * initial state (when the workload has one) ~ 0.1 * N(0, 1), fp32.
  * scale = K ** -0.5.
Casts to bf16 round to nearest even (torch's conversion).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    io_dtype: str            # "f32" or "bf16"
    B: int
    T: int                   # tokens per sequence (fixed-length) or packed total (varlen)
    H: int
    HV: int
    K: int
    V: int
    init_state: bool         # an initial state is read
    num_seqs: int = 0        # varlen: number of packed sequences (B must be 1)
    max_len: int = 0         # varlen: lengths uniform in [1, max_len]
    note: str = ""


# The five workloads: shapes and value distributions as stated for the method's
# forward (fp32 parity case, the headline bf16 case, long sequences, varlen
# packing, grouped value heads).
WORKLOADS = [
    Workload("fp32_T128_H2_K64", "f32", 1, 128, 2, 2, 64, 64, False,
             note="fp32 I/O, chunk semantics 64, no initial state"),
    Workload("bf16_T4096_H32_K128", "bf16", 1, 4096, 32, 32, 128, 128, False,
             note="headline: zero initial state (not read)"),
    Workload("bf16_B4_T16384_H32_K128", "bf16", 4, 16384, 32, 32, 128, 128, True,
             note="long sequences, initial state read"),
    Workload("bf16_varlen16_H32_K128", "bf16", 1, 0, 32, 32, 128, 128, True,
             num_seqs=16, max_len=8192, note="16 packed sequences, lengths U[1,8192]"),
    Workload("bf16_gva_B2_T32768_H8_HV32_K128", "bf16", 2, 32768, 8, 32, 128, 128, True,
             note="grouped value heads, G = 4"),
]


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    scale: float
    initial_state: torch.Tensor | None
    cu_seqlens: torch.Tensor | None
    io_dtype: str
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "Inputs":
        f = lambda t: None if t is None else t.to(device)
        return Inputs(f(self.q), f(self.k), f(self.v), f(self.g), f(self.beta), self.scale,
                      f(self.initial_state), f(self.cu_seqlens), self.io_dtype, dict(self.meta))

    @property
    def num_seqs(self) -> int:
        if self.cu_seqlens is not None:
            return int(self.cu_seqlens.numel() - 1)
        return int(self.q.shape[0])

    def tokens(self) -> int:
        return int(self.q.shape[0] * self.q.shape[1])


def _torch_dtype(io_dtype: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io_dtype]


def _l2norm(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float32) ** 2, axis=-1, keepdims=True, dtype=np.float32))
    return (x / n).astype(np.float32)


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    return (np.minimum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def varlen_lengths(rng: np.random.Generator, num_seqs: int, max_len: int) -> np.ndarray:
    return rng.integers(1, max_len + 1, size=num_seqs, dtype=np.int64)


def make_inputs(B: int, T: int, H: int, HV: int, K: int, V: int, io_dtype: str = "bf16",
                seed: int = 0, init_state: bool = False, lengths=None,
                g_scale: float = 1.0 / 8.0, gate: str = "logsigmoid", gate_value: float = -5.0) -> Inputs:
    """Draw one set of inputs.  ``lengths`` (a list of ints) selects varlen packing
    (then B must be 1 and T is ignored).  The decay g per (token, value head, key dim):
      gate="logsigmoid": g = g_scale * logsigmoid(N(0,1))  (g_scale = 1/8 in every stated
                         workload; 1 gives the unscaled gate)
      gate="bounded":    g = gate_value * sigmoid(N(0,1))  (a lower-bounded gate, gate_value
                         the bound, e.g. -5)
      gate="const":      g = gate_value everywhere (the same normal draw is still taken, so
                         the other tensors do not change with the gate)."""
    rng = np.random.default_rng(seed)
    cu = None
    if lengths is not None:
        assert B == 1
        lengths = np.asarray(lengths, dtype=np.int64)
        cu = np.zeros(len(lengths) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lengths)
        T = int(cu[-1])
    n_seq = len(lengths) if lengths is not None else B
    q = _l2norm(rng.standard_normal((B, T, H, K), dtype=np.float32))
    k = _l2norm(rng.standard_normal((B, T, H, K), dtype=np.float32))
    v = rng.standard_normal((B, T, HV, V), dtype=np.float32)
    gn = rng.standard_normal((B, T, HV, K), dtype=np.float32)
    if gate == "logsigmoid":
        g = _logsigmoid(gn) * np.float32(g_scale)
    elif gate == "bounded":
        g = np.float32(gate_value) * _sigmoid(gn)
    elif gate == "const":
        g = np.full_like(gn, np.float32(gate_value))
    else:
        raise ValueError(f"unknown gate {gate!r}")
    beta = _sigmoid(rng.standard_normal((B, T, HV), dtype=np.float32))
    s0 = None
    if init_state:
        s0 = (rng.standard_normal((n_seq, HV, K, V), dtype=np.float32) * np.float32(0.1))
    dt = _torch_dtype(io_dtype)
    return Inputs(
        q=torch.from_numpy(q).to(dt), k=torch.from_numpy(k).to(dt), v=torch.from_numpy(v).to(dt),
        g=torch.from_numpy(g.astype(np.float32)), beta=torch.from_numpy(beta),
        scale=float(K) ** -0.5,
        initial_state=None if s0 is None else torch.from_numpy(s0),
        cu_seqlens=None if cu is None else torch.from_numpy(cu.astype(np.int32)),
        io_dtype=io_dtype)


@dataclass
class RawInputs:
    """Raw projections for the forward with the pre-stage fused in."""
    q: torch.Tensor          # [B, T, H, K] unnormalised
    k: torch.Tensor
    v: torch.Tensor
    g_raw: torch.Tensor      # [B, T, HV, K] bf16 gate input
    beta_raw: torch.Tensor   # [B, T, HV] fp32
    A_log: torch.Tensor      # [HV] fp32
    dt_bias: torch.Tensor    # [HV, K] fp32
    scale: float
    initial_state: torch.Tensor | None
    cu_seqlens: torch.Tensor | None
    meta: dict = field(default_factory=dict)

    def to(self, device) -> "RawInputs":
        f = lambda t: None if t is None else t.to(device)
        return RawInputs(f(self.q), f(self.k), f(self.v), f(self.g_raw), f(self.beta_raw), f(self.A_log),
                         f(self.dt_bias), self.scale, f(self.initial_state), f(self.cu_seqlens), dict(self.meta))

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens.numel() - 1) if self.cu_seqlens is not None else int(self.q.shape[0])

    def tokens(self) -> int:
        return int(self.q.shape[0] * self.q.shape[1])


def make_raw_inputs(B: int, T: int, H: int, HV: int, K: int, V: int, seed: int = 0, init_state: bool = False,
                    lengths=None, param_scale: float = 0.1) -> RawInputs:
    """Raw projections (bf16 q, k, v and gate input) for the gated forward.  Recipe:
    numpy PCG64 seeded with `seed`; draw order q, k, v, g_raw, beta_raw, A_log, dt_bias,
    initial state.  q, k, v, g_raw ~ N(0, 1) (q and k NOT normalised: the pre-stage
    does it), beta_raw ~ N(0, 1), A_log and dt_bias ~ param_scale * N(0, 1), initial
    state 0.1 N(0, 1).  With the bounded gate and lower bound -5 this gives
    g = -5 sigmoid(~N(0, 1)) per element."""
    rng = np.random.default_rng(seed)
    cu = None
    if lengths is not None:
        assert B == 1
        lengths = np.asarray(lengths, dtype=np.int64)
        cu = np.zeros(len(lengths) + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lengths)
        T = int(cu[-1])
    n_seq = len(lengths) if lengths is not None else B
    q = rng.standard_normal((B, T, H, K), dtype=np.float32)
    k = rng.standard_normal((B, T, H, K), dtype=np.float32)
    v = rng.standard_normal((B, T, HV, V), dtype=np.float32)
    g = rng.standard_normal((B, T, HV, K), dtype=np.float32)
    beta = rng.standard_normal((B, T, HV), dtype=np.float32)
    A_log = rng.standard_normal(HV, dtype=np.float32) * np.float32(param_scale)
    dt = rng.standard_normal((HV, K), dtype=np.float32) * np.float32(param_scale)
    s0 = rng.standard_normal((n_seq, HV, K, V), dtype=np.float32) * np.float32(0.1) if init_state else None
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    return RawInputs(bf(q), bf(k), bf(v), bf(g), torch.from_numpy(beta), torch.from_numpy(A_log), torch.from_numpy(dt),
                     float(K) ** -0.5, None if s0 is None else torch.from_numpy(s0),
                     None if cu is None else torch.from_numpy(cu.astype(np.int32)))


def workload_raw_inputs(index: int) -> RawInputs:
    """Raw projections with the shapes of workload `index` (for the gated forward)."""
    w = WORKLOADS[index]
    lengths = None
    if w.num_seqs:
        lengths = varlen_lengths(np.random.default_rng(1000 + index), w.num_seqs, w.max_len)
    x = make_raw_inputs(w.B, w.T, w.H, w.HV, w.K, w.V, seed=index, init_state=w.init_state, lengths=lengths)
    x.meta["workload"] = w.name + "_gated"
    return x


def workload_inputs(index: int) -> Inputs:
    """Inputs of workload ``index`` (0..4), seeded with the index."""
    w = WORKLOADS[index]
    lengths = None
    if w.num_seqs:
        lengths = varlen_lengths(np.random.default_rng(1000 + index), w.num_seqs, w.max_len)
    x = make_inputs(w.B, w.T, w.H, w.HV, w.K, w.V, w.io_dtype, seed=index,
                    init_state=w.init_state, lengths=lengths)
    x.meta["workload"] = w.name
    return x


def algorithmic_bytes(x: Inputs, final_state: bool = True) -> int:
    """Bytes the forward must move at least once: every input read once, o and
    the final state written once."""
    el = lambda t: 0 if t is None else t.numel() * t.element_size()
    out = x.v.numel() * x.v.element_size()
    HV, K, V = x.v.shape[2], x.q.shape[3], x.v.shape[3]
    fs = x.num_seqs * HV * K * V * 4 if final_state else 0
    return (el(x.q) + el(x.k) + el(x.v) + el(x.g) + el(x.beta) + el(x.initial_state)
            + el(x.cu_seqlens) + out + fs)


def flops_convention(x: Inputs, C: int = 64) -> int:
    """Flop count used for reporting: per token and value head
    6*K*V + 6*C*K + 4*C*V at the nominal chunk C = 64 (triangular halves counted
    in full)."""
    HV, K, V = x.v.shape[2], x.q.shape[3], x.v.shape[3]
    return x.tokens() * HV * (6 * K * V + 6 * C * K + 4 * C * V)
