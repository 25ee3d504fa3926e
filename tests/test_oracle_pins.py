"""Pins for the fp64 oracle, checked against things other than the oracle itself.

The pages print no numeric example for KDA (their formula sections lost their
images), so the pins are: a brute-force evaluation over the full (K*V)-dimensional
state space, closed forms, the textbook delta rule, a hand-computed scalar
fixture, and invariants the method must satisfy.  Each is chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign, beta on the wrong
side, exp2 for exp, a transposed operand, a wrong GVA map) fails at least one.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(rng, B, T, H, HV, K, V, g_scale=0.125, s0=False, n_seq=None):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V))
    g = -np.abs(rng.standard_normal((B, T, HV, K))) * g_scale * 4
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, HV))))
    S0 = rng.standard_normal((n_seq or B, HV, K, V)) * 0.5 if s0 else None
    f = lambda a: None if a is None else a.astype(np.float32)
    return f(q), f(k), f(v), f(g), f(beta), f(S0)


def brute_force(q, k, v, g, beta, scale, S0=None):
    """Evaluate the recurrence as an affine map on vec(S) (row-major, K*V entries),
    building each token's transition with Kronecker products:
        vec(S_t) = kron((I - b k k^T) Diag(e^g), I_V) vec(S_{t-1}) + vec(b k v^T)
        o_t      = scale * kron(q^T, I_V) vec(S_t)."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    o = np.zeros((B, T, HV, V))
    S = np.zeros((B, HV, K, V))
    IV = np.eye(V)
    for b in range(B):
        for h in range(HV):
            s = np.zeros(K * V) if S0 is None else S0[b, h].astype(np.float64).reshape(-1)
            for t in range(T):
                kt = k[b, t, h // G].astype(np.float64)
                qt = q[b, t, h // G].astype(np.float64)
                bt = float(beta[b, t, h])
                left = (np.eye(K) - bt * np.outer(kt, kt)) @ np.diag(np.exp(g[b, t, h].astype(np.float64)))
                s = np.kron(left, IV) @ s + np.outer(bt * kt, v[b, t, h].astype(np.float64)).reshape(-1)
                o[b, t, h] = scale * (np.kron(qt[None, :], IV) @ s)
            S[b, h] = s.reshape(K, V)
    return o, S


@pytest.mark.parametrize("form,chunk", [("recurrent", 1), ("chunked", 1), ("chunked", 3),
                                        ("chunked", 4), ("chunked", 64)])
def test_brute_force_kronecker(form, chunk):
    rng = np.random.default_rng(11)
    B, T, H, HV, K, V = 2, 9, 1, 2, 3, 2
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    scale = 0.7
    o_ref, S_ref = brute_force(q, k, v, g, beta, scale, S0)
    o, S = oracle.forward(q, k, v, g, beta, scale, initial_state=S0, form=form, chunk=chunk)
    assert np.abs(o - o_ref).max() <= 1e-12 * max(1.0, np.abs(o_ref).max())
    assert np.abs(S - S_ref).max() <= 1e-12 * max(1.0, np.abs(S_ref).max())


@pytest.mark.parametrize("T", [1, 17, 64, 130])
def test_chunk_size_independence(T):
    rng = np.random.default_rng(T)
    B, H, HV, K, V = 1, 2, 2, 8, 5
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    o_r, S_r = oracle.forward(q, k, v, g, beta, 0.5, S0, form="recurrent")
    for C in (1, 2, 3, 16, 64):
        o_c, S_c = oracle.forward(q, k, v, g, beta, 0.5, S0, form="chunked", chunk=C)
        assert np.abs(o_c - o_r).max() <= 1e-12 * np.abs(o_r).max()
        assert np.abs(S_c - S_r).max() <= 1e-12 * np.abs(S_r).max()


def test_tri_inverse_identity_and_neumann():
    rng = np.random.default_rng(3)
    for n in (1, 5, 16, 64):
        M = np.tril(rng.standard_normal((n, n)) * 0.3, -1)
        T = oracle.tri_inverse(M)
        assert np.abs((np.eye(n) + M) @ T - np.eye(n)).max() <= 1e-12
        assert np.allclose(T, np.tril(T))
        assert np.allclose(np.diag(T), 1.0)
    # 16 x 16: the inverse equals the finite Neumann product (M is nilpotent, M^16 = 0):
    # (I + M)^{-1} = (I - M)(I + M^2)(I + M^4)(I + M^8)
    M = np.tril(rng.standard_normal((16, 16)) * 0.3, -1)
    I = np.eye(16)
    M2 = M @ M
    M4 = M2 @ M2
    M8 = M4 @ M4
    neumann = (I - M) @ (I + M2) @ (I + M4) @ (I + M8)
    T = oracle.tri_inverse(M)
    assert np.abs(T - neumann).max() <= 1e-12 * np.abs(neumann).max()


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_beta_zero_is_pure_decay(form):
    rng = np.random.default_rng(5)
    B, T, H, HV, K, V = 1, 70, 1, 1, 6, 4
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    beta[:] = 0
    o, S = oracle.forward(q, k, v, g, beta, 0.3, S0, form=form, chunk=16)
    G = np.cumsum(g[0, :, 0].astype(np.float64), axis=0)          # [T, K]
    St = np.exp(G)[:, :, None] * S0[0, 0][None].astype(np.float64)  # [T, K, V]
    o_ref = 0.3 * np.einsum("tk,tkv->tv", q[0, :, 0].astype(np.float64), St)
    assert np.abs(o[0, :, 0] - o_ref).max() <= 1e-12 * np.abs(o_ref).max()
    assert np.abs(S[0, 0] - St[-1]).max() <= 1e-12 * np.abs(St[-1]).max()


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_delta_rule_exact_retrieval(form):
    """g = 0, beta = 1, unit-norm keys: the plain delta rule writes v_t exactly
    under k_t, so reading with q_t = k_t returns v_t (o_t = S_t^T k_t)."""
    rng = np.random.default_rng(6)
    B, T, H, HV, K, V = 1, 40, 1, 1, 8, 5
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    # keys with exactly unit norm in binary floating point: +-1/2 on four of the
    # eight coordinates
    k[:] = 0
    for t in range(T):
        idx = rng.choice(K, size=4, replace=False)
        k[0, t, 0, idx] = rng.choice([-0.5, 0.5], size=4)
    g[:] = 0
    beta[:] = 1
    o, _ = oracle.forward(k, k, v, g, beta, 1.0, S0, form=form, chunk=7)
    assert np.abs(o - v.astype(np.float64)).max() <= 1e-10


def test_delta_rule_matches_textbook_update():
    """g = 0: each step is the textbook delta-rule update S += beta k (v - S^T k)^T."""
    rng = np.random.default_rng(7)
    T, K, V = 25, 6, 3
    q, k, v, g, beta, _ = rand_inputs(rng, 1, T, 1, 1, K, V)
    g[:] = 0
    o, S = oracle.forward(q, k, v, g, beta, 1.0, None, form="chunked", chunk=8)
    Sr = np.zeros((K, V))
    for t in range(T):
        kt, vt, qt = (x[0, t, 0].astype(np.float64) for x in (k, v, q))
        pred = Sr.T @ kt
        Sr = Sr + float(beta[0, t, 0]) * np.outer(kt, vt - pred)
        assert np.allclose(o[0, t, 0], Sr.T @ qt, rtol=0, atol=1e-12)
    assert np.allclose(S[0, 0], Sr, rtol=0, atol=1e-12)


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_scalar_golden_fixture(form):
    rows = np.loadtxt(os.path.join(GOLDEN, "scalar_k1v1.txt"), comments="#")
    T = rows.shape[0]
    q = rows[:, 0].reshape(1, T, 1, 1).astype(np.float32)
    k = rows[:, 1].reshape(1, T, 1, 1).astype(np.float32)
    v = rows[:, 2].reshape(1, T, 1, 1).astype(np.float32)
    g = np.log(rows[:, 3]).reshape(1, T, 1, 1).astype(np.float32)
    beta = rows[:, 4].reshape(1, T, 1).astype(np.float32)
    o, S = oracle.forward(q, k, v, g, beta, 1.0, None, form=form, chunk=3)
    np.testing.assert_allclose(o[0, :, 0, 0], rows[:, 6], rtol=1e-7, atol=1e-7)
    np.testing.assert_allclose(S[0, 0, 0, 0], rows[-1, 5], rtol=1e-7, atol=1e-7)


@pytest.mark.parametrize("form", ["recurrent", "chunked"])
def test_split_sequence_continuity(form):
    rng = np.random.default_rng(8)
    B, T, H, HV, K, V = 1, 100, 1, 2, 8, 6
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    o, S = oracle.forward(q, k, v, g, beta, 0.4, S0, form=form, chunk=16)
    m = 37
    sl = lambda a, a0, a1: a[:, a0:a1]
    o1, S1 = oracle.forward(*(sl(a, 0, m) for a in (q, k, v, g, beta)), 0.4, S0, form=form, chunk=16)
    o2, S2 = oracle.forward(*(sl(a, m, T) for a in (q, k, v, g, beta)), 0.4, S1.astype(np.float32),
                            form=form, chunk=16)
    # the carried state is rounded to fp32 when passed back in; compare loosely
    assert np.abs(np.concatenate([o1, o2], axis=1) - o).max() <= 1e-6 * np.abs(o).max()
    assert np.abs(S2 - S).max() <= 1e-6 * np.abs(S).max()


def test_gva_equals_repeated_heads():
    rng = np.random.default_rng(9)
    B, T, H, HV, K, V = 1, 33, 2, 8, 4, 3
    q, k, v, g, beta, S0 = rand_inputs(rng, B, T, H, HV, K, V, s0=True)
    o, S = oracle.forward(q, k, v, g, beta, 0.5, S0, form="chunked", chunk=8)
    G = HV // H
    qr, kr = np.repeat(q, G, axis=2), np.repeat(k, G, axis=2)   # key head hv // G
    o2, S2 = oracle.forward(qr, kr, v, g, beta, 0.5, S0, form="recurrent")
    assert np.abs(o - o2).max() <= 1e-12 * np.abs(o).max()
    assert np.abs(S - S2).max() <= 1e-12 * np.abs(S).max()


def test_varlen_equals_separate_calls_and_empty_sequence():
    rng = np.random.default_rng(10)
    lens = [5, 0, 19, 1, 40]
    T = sum(lens)
    H, HV, K, V = 1, 2, 4, 3
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, T, H, HV, K, V, s0=True, n_seq=len(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, S = oracle.forward(q, k, v, g, beta, 0.5, S0, cu_seqlens=cu, form="chunked", chunk=16)
    for i, L in enumerate(lens):
        a0, a1 = cu[i], cu[i + 1]
        if L == 0:
            assert np.array_equal(S[i], S0[i].astype(np.float64))
            continue
        oi, Si = oracle.forward(*(x[:, a0:a1] for x in (q, k, v, g, beta)), 0.5, S0[i:i + 1],
                                form="recurrent")
        assert np.abs(o[:, a0:a1] - oi).max() <= 1e-12 * np.abs(oi).max()
        assert np.abs(S[i] - Si[0]).max() <= 1e-12 * np.abs(Si).max()


def test_zero_padded_row_is_identity():
    """A row with k = 0 and g = 0 leaves the state unchanged (the reading used
    for rows past the end of a partial chunk)."""
    rng = np.random.default_rng(12)
    T, K, V = 10, 4, 3
    q, k, v, g, beta, S0 = rand_inputs(rng, 1, T, 1, 1, K, V, s0=True)
    _, S = oracle.forward(q, k, v, g, beta, 0.5, S0, form="recurrent")
    pad = lambda a, val: np.concatenate([a, np.full_like(a[:, :3], val)], axis=1)
    _, S2 = oracle.forward(pad(q, 1.0), pad(k, 0.0), pad(v, 1.0), pad(g, 0.0), pad(beta, 0.5),
                           0.5, S0, form="chunked", chunk=4)
    assert np.abs(S - S2).max() <= 1e-12 * np.abs(S).max()


# ---------------------------------------------------------------- pre-stage --
# The activations of the gated forward (q/k L2 normalisation, the bounded and the
# softplus gate, the beta sigmoid), pinned by closed forms chosen so that a slip
# (eps outside the root, the norm over the wrong axis, A_log not exponentiated,
# dt_bias added after the scale, dt_bias transposed, the wrong head's parameters)
# changes a checked value.

def _prestage(q=None, k=None, g=None, b=None, A_log=None, dt=None, gate="bounded", lb=-5.0,
              B=1, T=2, H=1, HV=2, K=4):
    z = lambda *s: np.zeros(s, dtype=np.float32)
    q = z(B, T, H, K) if q is None else q
    k = z(B, T, H, K) if k is None else k
    g = z(B, T, HV, K) if g is None else g
    b = z(B, T, HV) if b is None else b
    A_log = z(HV) if A_log is None else A_log
    dt = z(HV, K) if dt is None else dt
    return oracle.prestage(q, k, g, b, A_log, dt, gate=gate, lower_bound=lb)


def test_prestage_l2_norm_closed_form():
    q = np.zeros((1, 2, 2, 4), dtype=np.float32)
    q[0, 0, 0, 2] = 3.0                       # one non-zero entry: 3 / sqrt(9 + 1e-6)
    q[0, 0, 1] = [1.0, 2.0, 2.0, 4.0]         # |q|^2 = 25, the other key head
    q[0, 1, 0] = [1e-4, 0.0, 0.0, 0.0]        # |q|^2 = 1e-8, well below eps
    qn, kn, _, _ = _prestage(q=q, k=q * 7, H=2, HV=2)
    assert qn[0, 0, 0, 2] == pytest.approx(3.0 / np.sqrt(9.0 + 1e-6), rel=1e-15)
    assert np.count_nonzero(qn[0, 0, 0]) == 1
    np.testing.assert_allclose(qn[0, 0, 1], np.array([1, 2, 2, 4]) / np.sqrt(25.0 + 1e-6), rtol=1e-15)
    assert qn[0, 1, 0, 0] == pytest.approx(1e-4 / np.sqrt(1e-8 + 1e-6), rel=1e-6)   # eps dominates: ~0.0995
    assert np.all(qn[0, 1, 1] == 0.0)        # an all-zero row stays zero
    np.testing.assert_allclose(kn[0, 0, 1], 7 * np.array([1, 2, 2, 4]) / np.sqrt(49 * 25.0 + 1e-6), rtol=1e-15)


def test_prestage_beta_sigmoid():
    b = np.array([[[0.0, np.log(3.0)], [-np.log(3.0), 40.0]]], dtype=np.float32)
    _, _, _, beta = _prestage(b=b)
    assert beta[0, 0, 0] == 0.5
    assert beta[0, 0, 1] == pytest.approx(0.75, rel=1e-7)     # 1 / (1 + 1/3); ln 3 rounded to fp32
    assert beta[0, 1, 0] == pytest.approx(0.25, rel=1e-6)
    assert beta[0, 1, 1] == pytest.approx(1.0, abs=1e-17)


def test_prestage_bounded_gate_closed_forms():
    HV, K = 2, 4
    ln3 = np.log(3.0)
    A_log = np.array([np.log(2.0), 0.0], dtype=np.float32)           # a = 2 for head 0, a = 1 for head 1
    dt = np.zeros((HV, K), dtype=np.float32)
    dt[0] = [ln3 / 2, 0.0, 0.0, -ln3 / 2]                             # per dim, head 0 only
    g = np.zeros((1, 2, HV, K), dtype=np.float32)
    g[0, 1, 0, 1] = ln3 / 2
    g[0, 1, 1, 2] = ln3
    g[0, 1, 1, 3] = 60.0
    _, _, ga, _ = _prestage(g=g, A_log=A_log, dt=dt, lb=-5.0)
    # token 0: sigmoid(a * dt): head 0 dims 0 and 3 -> sigmoid(+-ln 3) = 3/4, 1/4; else 1/2
    np.testing.assert_allclose(ga[0, 0, 0], [-3.75, -2.5, -2.5, -1.25], rtol=1e-6)
    np.testing.assert_allclose(ga[0, 0, 1], [-2.5] * 4, rtol=1e-15)
    # token 1: head 0 dim 1 -> a * (ln3/2 + 0) = ln 3; head 1 dim 2 -> ln 3, dim 3 -> 60 (saturates at lb)
    assert ga[0, 1, 0, 1] == pytest.approx(-3.75, rel=1e-6)
    assert ga[0, 1, 1, 2] == pytest.approx(-3.75, rel=1e-6)
    assert ga[0, 1, 1, 3] == pytest.approx(-5.0, rel=1e-15)
    assert np.all(ga <= 0.0) and np.all(ga >= -5.0)


def test_prestage_softplus_gate_closed_forms():
    HV, K = 2, 4
    A_log = np.array([np.log(2.0), -50.0], dtype=np.float32)         # a = 2 (to fp32 rounding); a ~ 2e-22
    a = np.exp(np.float64(A_log[0]))                                   # exactly what the oracle is handed
    x1 = np.float64(np.float32(np.log(np.e - 1.0)))
    g = np.zeros((1, 2, HV, K), dtype=np.float32)
    g[0, 0, 0] = [0.0, x1, 40.0, -40.0]
    g[0, 1, 1] = [100.0, 0.0, 0.0, 0.0]
    _, _, ga, _ = _prestage(g=g, A_log=A_log, gate="softplus")
    assert abs(a - 2.0) < 1e-8
    assert ga[0, 0, 0, 0] == pytest.approx(-a * np.log(2.0), rel=1e-15)       # softplus(0) = ln 2
    assert ga[0, 0, 0, 1] == pytest.approx(-a * np.log(np.exp(x1) + 1.0), rel=1e-14)
    assert ga[0, 0, 0, 1] == pytest.approx(-2.0, rel=1e-7)                     # softplus(ln(e - 1)) = 1
    assert ga[0, 0, 0, 2] == pytest.approx(-a * 40.0, rel=1e-15)               # softplus(x) = x + O(e^-x)
    assert ga[0, 0, 0, 3] == pytest.approx(-a * np.exp(-40.0), rel=1e-12)     # softplus(x) = e^x + O(e^2x)
    assert abs(ga[0, 1, 1, 0]) < 1e-19                                          # a ~ 0: no decay at all


def test_gated_forward_reduces_to_exact_delta_rule_retrieval():
    """A vanishing gate (a = e^-60) and beta_raw = 40 (beta = 1 - 4e-18) make the gated
    forward the plain delta rule with unit-norm keys: after token t the state maps
    k^_t to v_t (up to the 1e-6 inside the norm), k^_t^T S_t = v_t^T."""
    rng = np.random.default_rng(21)
    B, T, H, HV, K, V = 1, 6, 1, 1, 8, 5
    q = rng.standard_normal((B, T, H, K)).astype(np.float32)
    k = rng.standard_normal((B, T, H, K)).astype(np.float32)
    v = rng.standard_normal((B, T, HV, V)).astype(np.float32)
    g = rng.standard_normal((B, T, HV, K)).astype(np.float32)
    b = np.full((B, T, HV), 40.0, dtype=np.float32)
    A_log = np.array([-60.0], dtype=np.float32)
    dt = np.zeros((HV, K), dtype=np.float32)
    for t in range(1, T + 1):
        sl = lambda a: a[:, :t]
        _, S = oracle.forward_gated(sl(q), sl(k), sl(v), sl(g), sl(b), A_log, dt, 1.0, gate="softplus")
        kn = k[0, t - 1, 0].astype(np.float64) / np.sqrt(np.sum(k[0, t - 1, 0].astype(np.float64) ** 2) + 1e-6)
        np.testing.assert_allclose(kn @ S[0, 0], v[0, t - 1, 0], atol=2e-5)


# ----------------------------------------------------------------- backward --
def _loss(q, k, v, g, b, s0, do, dsf, scale, cu=None):
    o, S = oracle.forward(q, k, v, g, b, scale, initial_state=s0, cu_seqlens=cu, form="recurrent")
    return float(np.sum(o * do) + np.sum(S * dsf))


@pytest.mark.parametrize("varlen", [False, True])
def test_backward_matches_central_differences(varlen):
    """Every input entry of a tiny problem (grouped value heads, an initial state, a
    final-state gradient; with varlen, an empty and a one-token sequence) against the
    central difference of the forward's loss sum <do, o> + <dS_final, S_final>.  The
    step is taken on the fp32 inputs the oracle reads, and divided by its exact size."""
    rng = np.random.default_rng(31)
    H, HV, K, V = 1, 2, 3, 2
    if varlen:
        lens = [3, 0, 1, 4]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        B, T, NS = 1, int(cu[-1]), len(lens)
    else:
        cu, B, T = None, 2, 5
        NS = B
    q, k, v, g, b, s0 = rand_inputs(rng, B, T, H, HV, K, V, g_scale=0.5, s0=True, n_seq=NS)
    b = np.clip(b, 0.05, 0.95).astype(np.float32)
    do = rng.standard_normal(v.shape).astype(np.float32)
    dsf = rng.standard_normal(s0.shape).astype(np.float32)
    scale = 0.7
    grads = oracle.backward(q, k, v, g, b, scale, do, d_final_state=dsf, initial_state=s0, cu_seqlens=cu)
    args = [q, k, v, g, b, s0]
    for ai, (arr, grad) in enumerate(zip(args, (grads[0], grads[1], grads[2], grads[3], grads[4], grads[5]))):
        for idx in np.ndindex(arr.shape):
            x0 = float(arr[idx])
            hstep = 1e-3 * max(1.0, abs(x0))
            up, dn = [a.copy() for a in args], [a.copy() for a in args]
            up[ai][idx] = np.float32(x0 + hstep)
            dn[ai][idx] = np.float32(x0 - hstep)
            step = float(up[ai][idx]) - float(dn[ai][idx])
            fd = (_loss(*up, do, dsf, scale, cu) - _loss(*dn, do, dsf, scale, cu)) / step
            assert abs(fd - grad[idx]) <= 2e-5 * max(1.0, abs(fd)), (ai, idx, fd, grad[idx])


def test_backward_of_an_empty_sequence_passes_the_state_gradient_through():
    q, k, v, g, b, s0 = rand_inputs(np.random.default_rng(3), 1, 0, 1, 1, 2, 2, s0=True)
    dsf = np.arange(4, dtype=np.float32).reshape(1, 1, 2, 2)
    *_, ds0 = oracle.backward(q, k, v, g, b, 1.0, np.zeros(v.shape, np.float32), d_final_state=dsf, initial_state=s0)
    assert np.array_equal(ds0, dsf.astype(np.float64))


@pytest.mark.parametrize("chunk", [1, 3, 16, 64])
def test_chunk_form_backward_equals_reverse_mode(chunk):
    """The oracle's two backward formulations -- reverse mode through the token
    recurrence (pinned above by central differences) and the chunk form (per-chunk
    recompute, a reverse sweep over the states, the triangular inverse's VJP) -- give the
    same gradients: grouped value heads, an initial state, a final-state gradient, a
    ragged last chunk, any chunk size."""
    rng = np.random.default_rng(40 + chunk)
    q, k, v, g, b, s0 = rand_inputs(rng, 2, 70, 2, 4, 8, 6, s0=True)
    do = rng.standard_normal(v.shape).astype(np.float32)
    dsf = rng.standard_normal(s0.shape).astype(np.float32)
    ref = oracle.backward(q, k, v, g, b, 0.6, do, d_final_state=dsf, initial_state=s0)
    got = oracle.backward_chunked(q, k, v, g, b, 0.6, do, d_final_state=dsf, initial_state=s0, chunk=chunk)
    for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), got, ref):
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-9 * np.abs(r).max(), err_msg=name)


def test_chunk_form_backward_varlen_and_strong_decay():
    """Packed sequences (an empty one, one shorter than a chunk, ragged ones) with the
    bounded gate at its limit (g = -5 per token: the chunk's cumulative decay reaches
    -320, beyond fp32's exponent range); the chunk form forms every exponent as a
    difference, so both formulations still agree."""
    rng = np.random.default_rng(47)
    lens = [0, 5, 64, 65, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, g, b, s0 = rand_inputs(rng, 1, int(cu[-1]), 1, 2, 8, 4, s0=True, n_seq=len(lens))
    g = np.full_like(g, -5.0)
    do = rng.standard_normal(v.shape).astype(np.float32)
    dsf = rng.standard_normal(s0.shape).astype(np.float32)
    ref = oracle.backward(q, k, v, g, b, 0.5, do, d_final_state=dsf, initial_state=s0, cu_seqlens=cu)
    got = oracle.backward_chunked(q, k, v, g, b, 0.5, do, d_final_state=dsf, initial_state=s0, cu_seqlens=cu)
    for name, a, r in zip(("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"), got, ref):
        assert np.all(np.isfinite(a)), name
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-9 * np.abs(r).max(), err_msg=name)
