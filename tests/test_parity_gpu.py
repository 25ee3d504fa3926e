"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.

Every workload is compared in full with the chunk kernels: the small and
headline ones in one oracle call, the large ones unit by unit, in the launch
configuration the benchmark times.  The token-recurrent kernel is compared on
sampled units of the large ones.
"""
import os

import numpy as np
import pytest
import torch

import kimi_delta_attention_gb300 as kda
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, check_all_units, check_units, np32, oracle_full, seq_bounds

pytestmark = pytest.mark.gpu


def _chunk_kernel(mode):
    """kda_chunk_fwd with the tensor-core kernel forced: "0" the cluster kernel,
    "1" the split kernel (chain and producer CTAs) where the unit count allows it."""
    def call(*args, **kw):
        old = os.environ.get("KDA_CHUNK_SPLIT")
        os.environ["KDA_CHUNK_SPLIT"] = mode
        try:
            return kda.kda_chunk_fwd(*args, **kw)
        finally:
            if old is None:
                del os.environ["KDA_CHUNK_SPLIT"]
            else:
                os.environ["KDA_CHUNK_SPLIT"] = old
    return call


ENTRIES = {"chunk": kda.kda_chunk_fwd, "chunk_cluster": _chunk_kernel("0"), "chunk_split": _chunk_kernel("1"),
           "recurrent": kda.kda_recurrent_fwd}
ALL = ["chunk", "chunk_cluster", "chunk_split", "recurrent"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def run(entry, x, **kw):
    d = x.to("cuda")
    o, S = ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                          cu_seqlens=d.cu_seqlens, **kw)
    torch.cuda.synchronize()
    return o, S


_cache = {}


def workload(i):
    if i not in _cache:
        _cache[i] = W.workload_inputs(i)
    return _cache[i]


@pytest.mark.parametrize("entry", ALL)
@pytest.mark.parametrize("idx", [0, 1])
def test_workload_full(entry, idx):
    x = workload(idx)
    o, S = run(entry, x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, x.io_dtype, f"w{idx} {entry}")


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_workload_every_unit(idx):
    """The large workloads at full size, in the launch configuration the benchmark
    uses (kda_chunk_fwd's own dispatch), compared with the oracle on every
    (sequence, value head) unit: o row by row and each final state."""
    x = workload(idx)
    o, S = run("chunk", x)
    check_all_units(x, o, S)


SAMPLED = {
    2: [(0, 0), (1, 9), (2, 20), (3, 31)],
    3: "all_seqs",
    4: [(0, 0), (0, 3), (1, 16), (1, 31)],
}


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_workload_sampled_recurrent(idx):
    """The token-recurrent kernel on the large workloads: sampled units."""
    x = workload(idx)
    o, S = run("recurrent", x)
    units = SAMPLED[idx]
    if units == "all_seqs":
        units = [(s, (5 * s) % x.v.shape[2]) for s in range(x.num_seqs)]
    check_units(x, o, S, units)
    # every output row and state is finite
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()


@pytest.mark.parametrize("entry", ["chunk_cluster", "chunk_split"])
def test_long_sequences_wrap_the_record_ring(entry):
    """256 chunks per unit: the per-unit record ring wraps many times, so the
    flow control between record producers and the chain is exercised."""
    x = W.make_inputs(1, 16384, 2, 4, 128, 128, "bf16", seed=12, init_state=True)
    o, S = run(entry, x)
    check_units(x, o, S, [(0, 0), (0, 3)])
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()


@pytest.mark.parametrize("entry", ALL)
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 100, 191, 257])
def test_ragged_lengths(entry, T):
    x = W.make_inputs(2, T, 2, 4, 128, 128, "bf16", seed=T, init_state=True)
    o, S = run(entry, x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", f"T={T}")


@pytest.mark.parametrize("entry", ["chunk", "recurrent"])
@pytest.mark.parametrize("KV", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_head_dims_and_dtypes(entry, KV, io):
    K, V = KV
    x = W.make_inputs(1, 150, 2, 2, K, V, io, seed=K + V, init_state=True)
    o, S = run(entry, x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, io, f"K={K} V={V} {io}")


@pytest.mark.parametrize("entry", ALL)
def test_varlen_with_empty_and_tiny_sequences(entry):
    lens = [0, 1, 64, 0, 77, 128, 3, 200, 0]
    x = W.make_inputs(1, 0, 2, 4, 128, 128, "bf16", seed=5, init_state=True, lengths=lens)
    o, S = run(entry, x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "varlen")
    s0 = x.initial_state.numpy()
    for i, L in enumerate(lens):
        if L == 0:  # an empty sequence hands its initial state through unchanged
            assert np.array_equal(S[i].cpu().numpy(), s0[i])


@pytest.mark.parametrize("entry", ALL)
def test_gva(entry):
    x = W.make_inputs(2, 130, 2, 8, 128, 128, "bf16", seed=3, init_state=True)
    o, S = run(entry, x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "gva")


@pytest.mark.parametrize("entry", ALL)
def test_empty_sequence_copies_state(entry):
    x = W.make_inputs(2, 0, 1, 2, 128, 128, "bf16", seed=1, init_state=True)
    o, S = run(entry, x)
    assert np.array_equal(S.cpu().numpy(), x.initial_state.numpy())
    x2 = W.make_inputs(1, 0, 1, 2, 64, 64, "bf16", seed=1, init_state=False)
    _, S2 = run(entry, x2)
    assert (S2 == 0).all()


@pytest.mark.parametrize("entry", ALL)
def test_in_place_state_and_no_final_state(entry):
    x = W.make_inputs(1, 200, 2, 2, 128, 128, "bf16", seed=4, init_state=True)
    o_ref, S_ref = oracle_full(x)
    d = x.to("cuda")
    st = d.initial_state.clone()
    o, S = ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=st, final_state=st)
    torch.cuda.synchronize()
    assert S.data_ptr() == st.data_ptr()
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "in-place")
    o2, S2 = ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                            output_final_state=False)
    torch.cuda.synchronize()
    assert S2 is None
    assert_close(o2.float().cpu().numpy(), None, o_ref, None, "bf16", "no final state")


@pytest.mark.parametrize("entry", ALL)
def test_split_sequence_continuity(entry):
    """Running [0, m) then [m, T) with the carried state equals one run over [0, T)."""
    x = W.make_inputs(1, 300, 2, 2, 128, 128, "bf16", seed=9, init_state=True)
    d = x.to("cuda")
    f = ENTRIES[entry]
    o, S = f(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state)
    m = 131
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, S1 = f(*(sl(t, 0, m) for t in (d.q, d.k, d.v, d.g, d.beta)), d.scale, initial_state=d.initial_state)
    o2, S2 = f(*(sl(t, m, 300) for t in (d.q, d.k, d.v, d.g, d.beta)), d.scale, initial_state=S1)
    torch.cuda.synchronize()
    oc = torch.cat([o1, o2], dim=1).float()
    assert (oc - o.float()).abs().max().item() <= 2e-2 * o.float().abs().max().item()
    assert ((S2 - S).norm() / S.norm()).item() <= 1e-2


@pytest.mark.parametrize("entry", ALL)
def test_beta_zero_pure_decay_full_size(entry):
    """Property at the headline size: with beta = 0 the state only decays,
    S_T = Diag(exp(sum_t g_t)) S_0.  The decay is scaled down (g = logsigmoid(N)/2000)
    so that exp(sum g) over 4096 tokens stays well inside fp32 range."""
    x = W.make_inputs(1, 4096, 4, 4, 128, 128, "bf16", seed=2, init_state=True, g_scale=1.0 / 2000)
    x.beta.zero_()
    d = x.to("cuda")
    _, S = ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state)
    torch.cuda.synchronize()
    G = x.g.double().sum(dim=1)[0]                          # [HV, K]
    S_ref = torch.exp(G)[:, :, None] * x.initial_state[0].double()
    err = ((S[0].double().cpu() - S_ref).norm() / S_ref.norm()).item()
    assert err <= 1e-2


@pytest.mark.parametrize("entry", ALL)
def test_bad_cu_seqlens_reports_device_status(entry):
    x = W.make_inputs(1, 0, 1, 2, 128, 128, "bf16", seed=6, init_state=True, lengths=[10, 20, 30])
    d = x.to("cuda")
    bad = torch.tensor([0, 40, 20, 60], dtype=torch.int32, device="cuda")   # decreasing
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(kda.make_shape(d.q, d.v, bad)), dtype=torch.uint8,
                     device="cuda")
    ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, cu_seqlens=bad,
                   workspace=ws)
    assert kda.kda_read_device_status(ws) == 7   # KDA_ERR_DEVICE_BOUNDS
    # the good call afterwards reports OK on the same workspace
    ENTRIES[entry](d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                   cu_seqlens=d.cu_seqlens, workspace=ws)
    assert kda.kda_read_device_status(ws) == 0


@pytest.mark.gpu
def test_call_on_another_stream_keeps_its_temporaries():
    """A call on a stream other than the current one, with the workspace left to the
    binding, gives the same result as a call on the current stream, even when the
    current stream allocates and overwrites memory right after the call returns."""
    x = W.make_inputs(1, 1024, 4, 8, 128, 128, "bf16", seed=77, init_state=True)
    d = x.to("cuda")
    ref_o, ref_s = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    o, s = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state,
                             stream=side.cuda_stream)
    junk = [torch.full((1 << 22,), 7, dtype=torch.int32, device="cuda") for _ in range(16)]
    torch.cuda.synchronize()
    del junk
    assert torch.equal(o, ref_o) and torch.equal(s, ref_s)


def test_split_kernel_over_several_launches():
    """More units than one split launch holds: launches of whole sequences on the same
    workspace (the status word gathers every launch's report)."""
    x = W.make_inputs(3, 1100, 2, 16, 128, 128, "bf16", seed=21, init_state=True)   # 48 units, 18 chunks
    d = x.to("cuda")
    shape = kda.make_shape(d.q, d.v)
    assert kda.kda_chunk_fwd_kernel_name(shape) == "kda_chunk_split_kernel"
    assert kda.kda_chunk_fwd_kernel_launches(shape) >= 2
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o, S = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == 0
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "split launches")


def test_split_kernel_launches_varlen():
    """Packed sequences of mixed lengths (empty ones included), the split kernel forced:
    several launches of whole sequences."""
    lens = [0, 1, 300, 64, 777, 129, 2, 1000, 65]
    x = W.make_inputs(1, 0, 2, 8, 128, 128, "bf16", seed=22, init_state=True, lengths=lens)   # 72 units
    o, S = run("chunk_split", x)
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", "split launches varlen")
    s0 = x.initial_state.numpy()
    assert np.array_equal(S[0].cpu().numpy(), s0[0])
