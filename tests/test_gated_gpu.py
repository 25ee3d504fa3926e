"""GPU parity of kda_chunk_fwd_gated: the chunked forward with the pre-stage (q/k
L2 normalisation, bounded or softplus gate on a bf16 gate input, beta sigmoid)
fused into the chunk kernels, against the oracle's fp64 pre-stage followed by its
token recurrence, on the exact bytes handed to the GPU."""
import os

import numpy as np
import pytest
import torch

import kimi_delta_attention_gb300 as kda
import oracle
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def oracle_gated(x, gate, lb):
    return oracle.forward_gated(np32(x.q), np32(x.k), np32(x.v), np32(x.g_raw), np32(x.beta_raw), np32(x.A_log),
                                np32(x.dt_bias), x.scale, gate=gate, lower_bound=lb,
                                initial_state=np32(x.initial_state),
                                cu_seqlens=None if x.cu_seqlens is None else x.cu_seqlens.numpy(), form="recurrent")


def run(x, gate, lb, split, ws=None):
    d = x.to("cuda")
    old = os.environ.get("KDA_CHUNK_SPLIT")
    try:
        if split is not None:
            os.environ["KDA_CHUNK_SPLIT"] = split
        o, S = kda.kda_chunk_fwd_gated(d.q, d.k, d.v, d.g_raw, d.beta_raw, d.A_log, d.dt_bias, gate=gate,
                                       lower_bound=lb, scale=d.scale, initial_state=d.initial_state,
                                       cu_seqlens=d.cu_seqlens, workspace=ws)
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("KDA_CHUNK_SPLIT", None)
        else:
            os.environ["KDA_CHUNK_SPLIT"] = old
    return o, S


@pytest.mark.parametrize("split", ["0", "1"])
@pytest.mark.parametrize("gate,lb", [("bounded", -5.0), ("bounded", -1.0), ("softplus", 0.0)])
def test_gated_matches_oracle(split, gate, lb):
    x = W.make_raw_inputs(2, 300, 2, 4, 128, 128, seed=51, init_state=True)   # GVA G = 2, ragged tail
    shape = kda.make_shape(x.q, x.v)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o, S = run(x, gate, lb, split, ws)
    assert kda.kda_read_device_status(ws) == 0
    o_ref, S_ref = oracle_gated(x, gate, lb)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", f"{gate} lb={lb} split={split}")


@pytest.mark.parametrize("split", ["0", "1"])
def test_gated_varlen_with_empty_sequences(split):
    x = W.make_raw_inputs(1, 0, 2, 4, 128, 128, seed=52, init_state=True, lengths=[0, 1, 65, 0, 200, 7])
    o, S = run(x, "bounded", -5.0, split)
    o_ref, S_ref = oracle_gated(x, "bounded", -5.0)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", f"gated varlen split={split}")
    s0 = x.initial_state.numpy()
    assert np.array_equal(S[0].cpu().numpy(), s0[0]) and np.array_equal(S[3].cpu().numpy(), s0[3])


def test_gated_headline_shape_every_unit():
    """The headline shape (B=1, T=4096, H=HV=32) through the default dispatch, all units."""
    x = W.workload_raw_inputs(1)
    o, S = run(x, "bounded", -5.0, None)
    o_ref, S_ref = oracle_gated(x, "bounded", -5.0)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "gated headline")


def test_gated_needs_the_tensor_core_shapes():
    x = W.make_raw_inputs(1, 64, 2, 2, 64, 64, seed=53)
    with pytest.raises(kda.KdaError) as e:
        run(x, "bounded", -5.0, None)
    assert e.value.code == 2
