"""kda_chunk_fwd_static_scratch: the forward for callers that cannot allocate
device memory (their host framework owns every allocation, or they must not pay
for cudaMalloc's implicit synchronisation on the hot path).  Its scratch lives in
a fixed array inside the library, so it must give the same results as
kda_chunk_fwd with a caller-provided workspace, and as the fp64 oracle, call
after call.

This file is collected last so that a stop-at-first-failure run has already
run every other test when it gets here."""
import ctypes

import numpy as np
import pytest
import torch

import kimi_delta_attention_gb300 as kda
from kimi_delta_attention_gb300 import _lib
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, oracle_full

# same bar as the parity tests (bf16 I/O): o relative to max|o|, state in Frobenius norm
O_TOL, S_TOL = 2e-2, 1e-2


def _rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).abs().max() / b.abs().max().clamp_min(1e-30)).item()


def _frob(a, b):
    a, b = a.double(), b.double()
    return ((a - b).norm() / b.norm().clamp_min(1e-30)).item()


def test_capacity_is_checked_on_the_host():
    """More than KDA_STATIC_SCRATCH_MAX_UNITS (sequence, value head) pairs is
    rejected before the library touches CUDA (fake, never-dereferenced pointers)."""
    kda.build()
    lib = _lib.load_library()
    P = ctypes.c_void_p
    fake = [P(0x100000 * (i + 1)) for i in range(7)]
    shape = _lib.KdaShape(1, 64, 33, 33, 128, 128, 0, _lib.KDA_BF16)   # 33 units
    status = ctypes.c_void_p()
    code = lib.kda_chunk_fwd_static_scratch(ctypes.byref(shape), fake[0], fake[1], fake[2], fake[3], fake[4],
                                            ctypes.c_float(0.088), None, None, fake[5], fake[6], None,
                                            ctypes.byref(status))
    assert code == 8 and kda.kda_status_string(code).startswith("more")


CASES = [
    dict(name="8 units, ragged tail", B=1, T=1000, H=8, HV=8, seed=21, init_state=False),
    dict(name="32 units (the limit), grouped value heads", B=2, T=700, H=2, HV=16, seed=22, init_state=True),
    dict(name="32 units, cluster kernel", B=2, T=700, H=2, HV=16, seed=23, init_state=True, split="0"),
    dict(name="varlen, 4 sequences x 8 value heads", lengths=[1, 130, 64, 300], H=4, HV=8, seed=24,
         init_state=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_static_scratch_matches_workspace_entry_two_calls_in_a_row(case, monkeypatch):
    """Two calls in a row through the C ABI; each is compared with kda_chunk_fwd on a
    caller-provided workspace and with the fp64 oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    if "split" in case:
        monkeypatch.setenv("KDA_CHUNK_SPLIT", case["split"])
    if "lengths" in case:
        x = W.make_inputs(1, 0, case["H"], case["HV"], 128, 128, "bf16", seed=case["seed"],
                          init_state=case["init_state"], lengths=case["lengths"])
    else:
        x = W.make_inputs(case["B"], case["T"], case["H"], case["HV"], 128, 128, "bf16", seed=case["seed"],
                          init_state=case["init_state"])
    o_or, s_or = oracle_full(x)
    d = x.to("cuda")
    o_ref, s_ref = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                                     cu_seqlens=d.cu_seqlens)
    for call in range(2):
        o, s, status_addr = kda.kda_chunk_fwd_static_scratch(d.q, d.k, d.v, d.g, d.beta, d.scale,
                                                             initial_state=d.initial_state,
                                                             cu_seqlens=d.cu_seqlens)
        torch.cuda.synchronize()
        assert status_addr
        assert _lib.load_library().kda_read_device_status(ctypes.c_void_p(status_addr), None) == 0
        assert torch.isfinite(o.float()).all()
        assert _rel(o, o_ref) <= O_TOL, (case["name"], call)
        assert _frob(s, s_ref) <= S_TOL, (case["name"], call)
        assert_close(o.float().cpu().numpy(), s.cpu().numpy(), o_or, s_or, "bf16", f"{case['name']} call {call}")


@pytest.mark.gpu
def test_static_scratch_rejects_too_many_units_on_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x = W.make_inputs(1, 64, 33, 33, 128, 128, "bf16", seed=3).to("cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_fwd_static_scratch(x.q, x.k, x.v, x.g, x.beta, x.scale)
    assert e.value.code == 8
