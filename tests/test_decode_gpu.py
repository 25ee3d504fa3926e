"""GPU parity of kda_decode, the recurrent step for inference: a few tokens per
sequence against a resident state updated in place, compared with the fp64
oracle's token recurrence (the state it returns is the decode's new state)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_gb300 as kda
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("KV", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_decode_matches_oracle(T, KV, io):
    K, V = KV
    x = W.make_inputs(6, T, 2, 8, K, V, io, seed=100 + T + K + V, init_state=True)   # 48 units, GVA G = 4
    d = x.to("cuda")
    state = d.initial_state.clone()
    o = kda.kda_decode(d.q, d.k, d.v, d.g, d.beta, state, d.scale)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), state.cpu().numpy(), o_ref, S_ref, io, f"decode T={T} K={K} V={V} {io}")


def test_decode_chain_equals_one_forward():
    """200 single-token steps carry the state exactly as one forward over the 200 tokens."""
    x = W.make_inputs(4, 200, 4, 8, 128, 128, "bf16", seed=7, init_state=True)
    d = x.to("cuda")
    state = d.initial_state.clone()
    outs = []
    for t in range(200):
        sl = lambda a: a[:, t:t + 1].contiguous()
        outs.append(kda.kda_decode(sl(d.q), sl(d.k), sl(d.v), sl(d.g), sl(d.beta), state, d.scale))
    torch.cuda.synchronize()
    o = torch.cat(outs, dim=1)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), state.cpu().numpy(), o_ref, S_ref, "bf16", "decode chain")
    o_c, S_c = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state)
    torch.cuda.synchronize()
    assert ((state - S_c).norm() / S_c.norm()).item() <= 1e-2


def test_decode_zero_tokens_keeps_the_state():
    x = W.make_inputs(2, 0, 2, 4, 128, 128, "bf16", seed=8, init_state=True)
    d = x.to("cuda")
    state = d.initial_state.clone()
    kda.kda_decode(d.q, d.k, d.v, d.g, d.beta, state, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(state, d.initial_state)
