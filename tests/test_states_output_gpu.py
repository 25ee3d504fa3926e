"""GPU parity of the two-pass forward: kda_chunk_states (the serial scan, writing the
state entering every chunk, h) and kda_chunk_output (every chunk's output from h, in
parallel), against the fp64 oracle run chunk by chunk with its state carried."""
import os

import numpy as np
import pytest
import torch

import kimi_delta_attention_gb300 as kda
import oracle
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, np32, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def oracle_chunk_states(x, C=64):
    """[B, HV, NT, K, V] float64: the oracle's state entering each chunk (its recurrence
    run over one chunk at a time, the state carried between the calls)."""
    q, k, v, g, b = (np32(t) for t in (x.q, x.k, x.v, x.g, x.beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    NT = (T + C - 1) // C
    S = np.zeros((B, HV, K, V)) if x.initial_state is None else np32(x.initial_state).astype(np.float64)
    hs = np.zeros((B, HV, NT, K, V))
    for n in range(NT):
        hs[:, :, n] = S
        sl = lambda a: a[:, n * C:(n + 1) * C]
        _, S = oracle.forward(sl(q), sl(k), sl(v), sl(g), sl(b), x.scale, initial_state=S.astype(np.float32),
                              form="recurrent")
    return hs, S


def with_split(mode, f):
    old = os.environ.get("KDA_CHUNK_SPLIT")
    os.environ["KDA_CHUNK_SPLIT"] = mode
    try:
        return f()
    finally:
        if old is None:
            os.environ.pop("KDA_CHUNK_SPLIT", None)
        else:
            os.environ["KDA_CHUNK_SPLIT"] = old


@pytest.mark.parametrize("split", ["0", "1"])
def test_states_match_the_oracle_chunk_by_chunk(split):
    x = W.make_inputs(2, 300, 2, 4, 128, 128, "bf16", seed=61, init_state=True)   # 5 chunks, tail of 44
    d = x.to("cuda")
    h, S = with_split(split, lambda: kda.kda_chunk_states(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state))
    torch.cuda.synchronize()
    h_ref, S_ref = oracle_chunk_states(x)
    assert h.shape == (2, 4, 5, 128, 128)
    hh = h.float().cpu().numpy()
    for b in range(2):
        for hv in range(4):
            for n in range(5):
                ref = h_ref[b, hv, n]
                err = np.linalg.norm(hh[b, hv, n] - ref) / np.linalg.norm(ref)
                assert err <= 1e-2, (b, hv, n, err)
    assert np.array_equal(hh[:, :, 0], np32(x.initial_state.to(torch.bfloat16)))   # h[0] is the initial state
    err = np.linalg.norm(S.cpu().numpy() - S_ref) / np.linalg.norm(S_ref)
    assert err <= 1e-2


@pytest.mark.parametrize("T", [64, 130, 300])
def test_output_from_oracle_states(T):
    """The output kernel alone: fed the oracle's states (bf16), its o matches the oracle's."""
    x = W.make_inputs(2, T, 2, 4, 128, 128, "bf16", seed=62 + T, init_state=True)
    h_ref, _ = oracle_chunk_states(x)
    d = x.to("cuda")
    h = torch.from_numpy(h_ref).to(torch.bfloat16).cuda()
    o = kda.kda_chunk_output(d.q, d.k, d.v, d.g, d.beta, h, d.scale)
    torch.cuda.synchronize()
    o_ref, _ = oracle_full(x)
    assert_close(o.float().cpu().numpy(), None, o_ref, None, "bf16", f"output T={T}")


@pytest.mark.parametrize("split", ["0", "1"])
def test_two_passes_equal_the_forward_at_the_headline_shape(split):
    x = W.workload_inputs(1)
    d = x.to("cuda")
    h, S = with_split(split, lambda: kda.kda_chunk_states(d.q, d.k, d.v, d.g, d.beta))
    o = kda.kda_chunk_output(d.q, d.k, d.v, d.g, d.beta, h, d.scale)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", f"two-pass split={split}")


def test_strong_decay_two_passes():
    x = W.make_inputs(1, 256, 2, 2, 128, 128, "bf16", seed=64, init_state=True, gate="bounded", gate_value=-5.0)
    d = x.to("cuda")
    h, S = kda.kda_chunk_states(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
    o = kda.kda_chunk_output(d.q, d.k, d.v, d.g, d.beta, h, d.scale)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "two-pass strong decay")


def test_unsupported_shapes():
    y = W.make_inputs(1, 64, 2, 2, 64, 64, "bf16", seed=66).to("cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_states(y.q, y.k, y.v, y.g, y.beta)
    assert e.value.code == 2
    with pytest.raises(kda.KdaError) as e:
        kda.kda_chunk_output(y.q, y.k, y.v, y.g, y.beta, torch.zeros(1, 2, 1, 64, 64, dtype=torch.bfloat16,
                                                                      device="cuda"), y.scale)
    assert e.value.code == 2
