"""Failure detection on the GPU without a fault: a wait limit the caller can shrink.

Every wait for work in the chunk kernels (a record, a ready flag, a product or a
tile not yet seen complete) gives up after the limit in KDA_WAIT_LIMIT_NS (2 s
by default); the role then records KDA_ERR_DEVICE_TIMEOUT in the status word,
drains the copies and products it already issued and returns.  With a 1 us
limit the first waits of a small problem run out: the call must still complete,
report the timeout, and leave the context and the workspace usable, so the next
call with the default limit succeeds and matches the oracle.
"""
import os

import pytest
import torch

import kimi_delta_attention_gb300 as kda
from kimi_delta_attention_gb300 import workloads as W
from kda_testutil import assert_close, oracle_full

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


class _env:
    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        for k, v in self.kv.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("split", ["0", "1"])
def test_short_wait_limit_reports_timeout_and_recovers(split):
    x = W.make_inputs(2, 256, 2, 4, 128, 128, "bf16", seed=41, init_state=True)   # 8 units, 4 chunks each
    d = x.to("cuda")
    shape = kda.make_shape(d.q, d.v)
    ws = torch.empty(kda.kda_chunk_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    with _env(KDA_CHUNK_SPLIT=split, KDA_WAIT_LIMIT_NS="1000"):
        assert kda.kda_chunk_fwd_kernel_name(shape) == ("kda_chunk_split_kernel" if split == "1"
                                                        else "kda_chunk_fused_kernel")
        kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, workspace=ws)
        torch.cuda.synchronize()
        assert kda.kda_read_device_status(ws) == KDA_ERR_DEVICE_TIMEOUT
    with _env(KDA_CHUNK_SPLIT=split, KDA_WAIT_LIMIT_NS=None):
        o, S = kda.kda_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, initial_state=d.initial_state, workspace=ws)
        torch.cuda.synchronize()
        assert kda.kda_read_device_status(ws) == 0
    o_ref, S_ref = oracle_full(x)
    assert_close(o.float().cpu().numpy(), S.cpu().numpy(), o_ref, S_ref, "bf16", f"after timeout, split={split}")


def test_backward_short_wait_limit_completes_and_recovers():
    """The chunk-form backward waits only on its own bulk copies and tcgen05 products (the
    state chains, the preparation's products), with the same limit; they end within
    microseconds, so a 1 us limit may or may not run out (mbarrier.try_wait suspends for a
    while before the limit is checked).  Either way the call must complete: status OK with
    the oracle's gradients, or a reported timeout after its drains; and the next call with
    the default limit must match the oracle."""
    import numpy as np
    import oracle
    from kda_testutil import np32
    x = W.make_inputs(1, 300, 2, 2, 128, 128, "bf16", seed=43, init_state=True)   # 5 chunks
    rng = np.random.default_rng(44)
    do = torch.from_numpy(rng.standard_normal(tuple(x.v.shape), dtype=np.float32)).to(torch.bfloat16)
    dfin = torch.from_numpy(rng.standard_normal(tuple(x.initial_state.shape), dtype=np.float32))
    d = x.to("cuda")
    shape = kda.make_shape(d.q, d.v)
    ws = torch.empty(kda.kda_backward_workspace_size(shape), dtype=torch.uint8, device="cuda")
    ref = oracle.backward(np32(x.q), np32(x.k), np32(x.v), np32(x.g), np32(x.beta), x.scale, np32(do),
                          d_final_state=np32(dfin), initial_state=np32(x.initial_state))

    def check(got, what):
        for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), got, ref):
            err = np.abs(a.cpu().numpy() - r).max() / max(np.abs(r).max(), 1e-30)
            assert err <= 1e-4, f"{what}: {name} error {err:.3e}"

    with _env(KDA_BACKWARD=None, KDA_WAIT_LIMIT_NS="1000"):
        got = kda.kda_backward(d.q, d.k, d.v, d.g, d.beta, do.cuda(), d.scale, initial_state=d.initial_state,
                               d_final_state=dfin.cuda(), workspace=ws)
        torch.cuda.synchronize()
        st = kda.kda_read_device_status(ws)
        assert st in (0, KDA_ERR_DEVICE_TIMEOUT)
        if st == 0:
            check(got, "1 us limit")
    with _env(KDA_BACKWARD=None, KDA_WAIT_LIMIT_NS=None):
        got = kda.kda_backward(d.q, d.k, d.v, d.g, d.beta, do.cuda(), d.scale, initial_state=d.initial_state,
                               d_final_state=dfin.cuda(), workspace=ws)
        torch.cuda.synchronize()
        assert kda.kda_read_device_status(ws) == 0
    check(got, "default limit after the short one")
