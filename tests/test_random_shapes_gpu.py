"""GPU parity on seeded random shapes, and the forward replayed from a CUDA graph.

The random sweep draws (B, T, H, G, K, V, dtype, packed lengths, initial state, gate)
from one seeded generator, so every run checks the same 24 problems: every kernel the
dispatch can pick (split, cluster, recurrent) against the fp64 oracle at the forward's
tolerances.  The graph test captures kda_chunk_fwd (its status-word memset and the
kernel launches) once and replays it on new inputs copied into the captured buffers.
"""
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


def _draw(i):
    rng = np.random.default_rng(9000 + i)
    K = int(rng.choice([64, 128], p=[0.25, 0.75]))
    V = int(rng.choice([64, 128], p=[0.25, 0.75]))
    io = "f32" if rng.random() < 0.2 else "bf16"
    H = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    init = bool(rng.random() < 0.6)
    gate = str(rng.choice(["logsigmoid", "bounded"], p=[0.7, 0.3]))
    if rng.random() < 0.35:
        lengths = [int(x) for x in rng.integers(0, 400, size=int(rng.integers(1, 6)))]
        return dict(B=1, T=0, H=H, HV=H * G, K=K, V=V, io=io, init=init, gate=gate, lengths=lengths)
    B = int(rng.integers(1, 4))
    T = int(rng.integers(1, 600))
    return dict(B=B, T=T, H=H, HV=H * G, K=K, V=V, io=io, init=init, gate=gate, lengths=None)


@pytest.mark.parametrize("i", range(24))
def test_random_shape_matches_oracle(i):
    c = _draw(i)
    x = W.make_inputs(c["B"], c["T"], c["H"], c["HV"], c["K"], c["V"], c["io"], seed=9100 + i,
                      init_state=c["init"], lengths=c["lengths"], gate=c["gate"], gate_value=-5.0)
    d = x.to("cuda")
    shape = kda.make_shape(d.q, d.v, d.cu_seqlens)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o, S = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                             cu_seqlens=d.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == 0
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, c["io"],
                 f"{c} via {kda.kda_chunk_fwd_kernel_name(shape)}")


@pytest.mark.parametrize("T", [4096, 300])
def test_forward_replayed_from_a_cuda_graph(T):
    """kda_chunk_fwd captured in a CUDA graph (stream capture of its memset and launches)
    and replayed: the replay on new inputs matches the oracle on those inputs."""
    shapes = dict(B=1, T=T, H=4, HV=8, K=128, V=128)
    x0 = W.make_inputs(shapes["B"], T, 4, 8, 128, 128, "bf16", seed=31, init_state=True)
    x1 = W.make_inputs(shapes["B"], T, 4, 8, 128, 128, "bf16", seed=32, init_state=True)
    d = x0.to("cuda")
    shape = kda.make_shape(d.q, d.v)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d.v)
    fin = torch.empty_like(d.initial_state)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # a warm call outside the capture (library set-up)
        kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, out=out,
                          final_state=fin, workspace=ws, stream=side.cuda_stream)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, out=out,
                          final_state=fin, workspace=ws, stream=torch.cuda.current_stream().cuda_stream)
    for x in (x1, x0):
        for name in ("q", "k", "v", "g", "beta", "initial_state"):
            getattr(d, name).copy_(getattr(x, name))
        graph.replay()
        torch.cuda.synchronize()
        assert kda.kda_read_device_status(ws) == 0
        o_ref, S_ref = oracle_full(x)
        assert_close(out.float().cpu().numpy(), fin.cpu().numpy(), o_ref, S_ref, "bf16", f"graph replay T={T}")
