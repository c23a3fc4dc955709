"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test states where its expectation comes from: a closed form of the
gate, the delta-rule overwrite property from the KDA row of the K3
architecture census, an explicit product of transition matrices, a textbook
special case, or an invariant that follows from the recurrence.  Together
they fail on a dropped term, a wrong sign, a transposed operand or a read
taken before instead of after the write.
"""
import json
import math

import numpy as np
import pytest

from conftest import golden_path

RTOL = 1e-12


def _rand_case(rng, T, H, dk, dv, N=1, nonzero_state=True, zscale=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    z = zscale * rng.standard_normal((T, H, dk))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    A = 0.5 * rng.standard_normal(H)
    S0 = 0.3 * rng.standard_normal((N, H, dk, dv)) if nonzero_state else None
    return q, k, v, z, beta, A, S0


def _unit(x, eps=1e-6):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def _gate_test_side(z, A):
    # Written independently of the oracle: g = -5 / (1 + exp(-e^A z)).
    return -5.0 / (1.0 + np.exp(-np.exp(A) * z))


def _close(a, b, tol=RTOL):
    a = np.asarray(a)
    b = np.asarray(b)
    scale = max(1.0, float(np.max(np.abs(b))))
    return float(np.max(np.abs(a - b))) <= tol * scale


# --------------------------------------------------------------------- gate
def test_gate_closed_forms(oracle_mod):
    data = json.load(open(golden_path("gate_closed_forms.json")))
    for c in data["cases"]:
        g = oracle_mod.gate(np.array([c["z"]]), c["A"])[0]
        assert abs(g - c["g"]) <= 1e-14, (c, g)


def test_gate_range_and_alpha_bounds(oracle_mod):
    rng = np.random.default_rng(1)
    z = np.concatenate([rng.standard_normal(10000) * 5, [1e4, -1e4, 0.0, 1e308, -1e308]])
    for A in (-3.0, -0.5, 0.0, 0.5, 2.0):
        g = oracle_mod.gate(z, A)
        assert np.all(g >= -5.0) and np.all(g <= 0.0)
        alpha = np.exp(g)
        assert np.all(alpha >= math.exp(-5.0)) and np.all(alpha <= 1.0)
        # g is monotone non-increasing in z
        order = np.argsort(z)
        assert np.all(np.diff(g[order]) <= 1e-15)


def test_tile_reciprocal_bound_fits_bf16():
    """16 tokens at g >= -5 give 1/Gamma <= e^80, inside the BF16 range."""
    data = json.load(open(golden_path("gate_closed_forms.json")))["tile_bound"]
    worst_log = -data["g_min"] * data["tokens"]
    assert worst_log == data["max_reciprocal_log"]
    assert math.exp(worst_log) < data["bf16_max"]
    # 17 tokens still fit, 18 do not: the bound is about tile length, not luck.
    assert math.exp(5.0 * 17) < data["bf16_max"] < math.exp(5.0 * 18)


# ---------------------------------------------------------------- overwrite
def test_overwrite_golden(oracle_mod):
    d = json.load(open(golden_path("overwrite_example.json")))
    T, dk, dv = len(d["v"]), d["d_k"], d["d_v"]
    q = np.array(d["q"]).reshape(T, 1, dk)
    k = np.array(d["k"]).reshape(T, 1, dk)
    v = np.array(d["v"]).reshape(T, 1, dv)
    beta = np.array(d["beta"]).reshape(T, 1)
    z = np.full((T, 1, dk), -1e4)          # sigmoid(-1e4) == 0 -> alpha == 1
    A = np.zeros(1)
    # k is exactly unit already; the in-op normalisation (with its 1e-6
    # epsilon) is pinned separately in test_scale_and_normalisation.
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, l2norm=False)
    assert _close(o[:, 0], d["expected_o"], 1e-12)
    assert not _close(o[1, 0], d["not_expected_o2"], 1e-3)
    assert _close(S[0, 0], d["expected_final_state"], 1e-12)


def test_delta_rule_readback(oracle_mod):
    """k_hat^T S_t = (1 - beta_t) k_hat^T Diag(alpha_t) S_{t-1} + beta_t v_t^T.

    With beta = 1 reading the key just written returns exactly v_t, whatever
    the decay and the earlier content (the overwrite property in general)."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 7, 2, 6, 5
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    k = _unit(k, eps=0.0)  # exactly unit keys; run without the in-op epsilon
    for beta_mode in ("one", "random"):
        b = np.ones_like(beta) if beta_mode == "one" else beta
        for t in range(1, T + 1):
            sl = slice(0, t)
            _, S_t, _ = oracle_mod.kda_reference(q[sl], k[sl], v[sl], z[sl], b[sl], A, S0,
                                                 l2norm=False)
            if t == 1:
                S_prev = S0
            else:
                _, S_prev, _ = oracle_mod.kda_reference(q[:t - 1], k[:t - 1], v[:t - 1],
                                                        z[:t - 1], b[:t - 1], A, S0,
                                                        l2norm=False)
            for h in range(H):
                kh = k[t - 1, h]
                alpha = np.exp(_gate_test_side(z[t - 1, h], A[h]))
                lhs = kh @ S_t[0, h]
                rhs = (1 - b[t - 1, h]) * (kh @ (alpha[:, None] * S_prev[0, h])) \
                    + b[t - 1, h] * v[t - 1, h]
                assert _close(lhs, rhs, 1e-11)


# ------------------------------------------------------------------ identity
def test_identity_alpha1_beta0(oracle_mod):
    rng = np.random.default_rng(3)
    T, H, dk, dv = 9, 3, 5, 4
    q, k, v, _, _, _, S0 = _rand_case(rng, T, H, dk, dv)
    z = np.full((T, H, dk), -1e4)
    A = np.zeros(H)
    beta = np.zeros((T, H))
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0)
    assert np.array_equal(S, S0)
    qh = _unit(q)
    for t in range(T):
        for h in range(H):
            assert _close(o[t, h], S0[0, h].T @ qh[t, h], 1e-13)


def test_decay_only_closed_form(oracle_mod):
    """beta = 0: S_t = Diag(e^{sum_{i<=t} g_i}) S0 and o_t = S_t^T q_hat_t."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 11, 2, 6, 3
    q, k, v, z, _, A, S0 = _rand_case(rng, T, H, dk, dv, zscale=2.0)
    beta = np.zeros((T, H))
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0)
    qh = _unit(q)
    for h in range(H):
        gam = np.cumsum(_gate_test_side(z[:, h], A[h]), axis=0)  # [T, dk]
        assert _close(S[0, h], np.exp(gam[-1])[:, None] * S0[0, h], 1e-12)
        for t in range(T):
            St = np.exp(gam[t])[:, None] * S0[0, h]
            assert _close(o[t, h], St.T @ qh[t, h], 1e-12)


# --------------------------------------------------------------- brute force
@pytest.mark.parametrize("T,dk,dv", [(1, 4, 3), (5, 4, 3), (8, 6, 5), (8, 3, 7)])
def test_brute_force_transition_products(oracle_mod, T, dk, dv):
    """Explicit M_t = (I - beta_t k_t k_t^T) Diag(alpha_t), then
    S_t = M_t...M_1 S0 + sum_i M_t...M_{i+1} beta_i k_i v_i^T,  o_t = S_t^T q_t."""
    rng = np.random.default_rng(10 + T + dk)
    H = 2
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0)
    qh, kh = _unit(q), _unit(k)
    for h in range(H):
        M = []
        for t in range(T):
            alpha = np.exp(_gate_test_side(z[t, h], A[h]))
            M.append((np.eye(dk) - beta[t, h] * np.outer(kh[t, h], kh[t, h])) @ np.diag(alpha))
        for t in range(T):
            P = np.eye(dk)
            for s in range(t, -1, -1):
                P = P @ M[s]
            St = P @ S0[0, h]
            for i in range(t + 1):
                Pi = np.eye(dk)
                for s in range(t, i, -1):
                    Pi = Pi @ M[s]
                St = St + Pi @ (beta[i, h] * np.outer(kh[i, h], v[i, h]))
            assert _close(o[t, h], St.T @ qh[t, h], 1e-12)
            if t == T - 1:
                assert _close(S[0, h], St, 1e-12)


# ------------------------------------------------------ chunked == recurrent
@pytest.mark.parametrize("C", [1, 3, 16, 64])
def test_chunked_form_equals_recurrent(oracle_mod, C):
    rng = np.random.default_rng(20 + C)
    lens = [50, 0, 37, 70]
    T, H, dk, dv = sum(lens), 2, 8, 6
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens), zscale=2.0)
    cu = np.concatenate([[0], np.cumsum(lens)])
    o_r, S_r, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu)
    o_c, S_c, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu, chunk=C)
    assert _close(o_c, o_r, 1e-10)
    assert _close(S_c, S_r, 1e-10)
    # the zero-length sequence returns its initial state
    assert np.array_equal(S_r[1], S0[1])


# ---------------------------------------------------------------- invariants
def test_linearity_in_v_and_state(oracle_mod):
    rng = np.random.default_rng(5)
    T, H, dk, dv = 12, 2, 5, 4
    q, k, v1, z, beta, A, S1 = _rand_case(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    a, b = 0.7, -1.9
    o1, F1, _ = oracle_mod.kda_reference(q, k, v1, z, beta, A, S1)
    o2, F2, _ = oracle_mod.kda_reference(q, k, v2, z, beta, A, S2)
    o3, F3, _ = oracle_mod.kda_reference(q, k, a * v1 + b * v2, z, beta, A, a * S1 + b * S2)
    assert _close(o3, a * o1 + b * o2, 1e-12)
    assert _close(F3, a * F1 + b * F2, 1e-12)


def test_value_column_permutation(oracle_mod):
    rng = np.random.default_rng(6)
    T, H, dk, dv = 10, 2, 4, 6
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    perm = rng.permutation(dv)
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0)
    op, Sp, _ = oracle_mod.kda_reference(q, k, v[..., perm], z, beta, A, S0[..., perm])
    assert _close(op, o[..., perm], 1e-13)
    assert _close(Sp, S[..., perm], 1e-13)


def test_textbook_causal_linear_attention(oracle_mod):
    """alpha = 1, beta = 1, orthonormal keys, zero state: o_t = sum_{i<=t} (q.k_i) v_i."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 6, 1, 8, 3
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:T].reshape(T, H, dk)
    q = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    z = np.full((T, H, dk), -1e4)
    A = np.zeros(H)
    beta = np.ones((T, H))
    o, _, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, l2norm=False)
    for t in range(T):
        ref = sum((q[t, 0] @ k[i, 0]) * v[i, 0] for i in range(t + 1))
        assert _close(o[t, 0], ref, 1e-12)


def test_contraction_bound(oracle_mod):
    """||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||: both factors of the
    transition have spectral norm <= 1 for unit k and beta in [0, 1]."""
    rng = np.random.default_rng(8)
    T, H, dk, dv = 16, 1, 6, 6
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    prev = np.linalg.norm(S0[0, 0], 2)
    for t in range(1, T + 1):
        _, S, _ = oracle_mod.kda_reference(q[:t], k[:t], v[:t], z[:t], beta[:t], A, S0)
        cur = np.linalg.norm(S[0, 0], 2)
        assert cur <= prev + beta[t - 1, 0] * np.linalg.norm(v[t - 1, 0]) + 1e-12
        prev = cur


def test_varlen_equals_separate_and_split_handoff(oracle_mod):
    rng = np.random.default_rng(9)
    lens = [13, 1, 20]
    T, H, dk, dv = sum(lens), 2, 5, 4
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        on, Sn, _ = oracle_mod.kda_reference(q[sl], k[sl], v[sl], z[sl], beta[sl], A, S0[n:n + 1])
        assert np.array_equal(on, o[sl])
        assert np.array_equal(Sn[0], S[n])
    # split the last sequence at 7 and hand the state over
    sl = slice(cu[2], cu[3])
    a = slice(cu[2], cu[2] + 7)
    b = slice(cu[2] + 7, cu[3])
    oa, Sa, _ = oracle_mod.kda_reference(q[a], k[a], v[a], z[a], beta[a], A, S0[2:3])
    ob, Sb, _ = oracle_mod.kda_reference(q[b], k[b], v[b], z[b], beta[b], A, Sa)
    assert np.array_equal(np.concatenate([oa, ob]), o[sl])
    assert np.array_equal(Sb[0], S[2])


def test_scale_and_normalisation(oracle_mod):
    """o is linear in `scale`; positive rescaling of raw q, k does not matter
    up to the 1e-6 epsilon under the root."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 9, 2, 7, 3
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    o1, S1, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, scale=1.0)
    o2, S2, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, scale=0.125)
    assert _close(o2, 0.125 * o1, 1e-13)
    assert np.array_equal(S1, S2)
    o3, S3, _ = oracle_mod.kda_reference(3.0 * q, 0.5 * k, v, z, beta, A, S0)
    assert _close(o3, o1, 1e-5) and _close(S3, S1, 1e-5)


def test_units_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(12)
    lens = [9, 14]
    T, H, dk, dv = sum(lens), 3, 4, 4
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=2)
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu)
    os_, Ss, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu, units=[(1, 2), (0, 0)])
    assert np.array_equal(os_[cu[1]:, 2], o[cu[1]:, 2])
    assert np.array_equal(os_[:cu[1], 0], o[:cu[1], 0])
    assert np.array_equal(Ss[1, 2], S[1, 2]) and np.array_equal(Ss[0, 0], S[0, 0])
    assert np.isnan(os_[:cu[1], 1]).all()


# ------------------------------------------------------------ state checkpoints
def test_checkpoints_are_prefix_final_states(oracle_mod):
    """Checkpoint m of sequence n is the final state of a run on its first
    m * interval tokens (a separate oracle run from the same initial state),
    and resuming from it reproduces the rest of the sequence; sequences
    shorter than the interval have none; a length that is a multiple of the
    interval ends with its final state."""
    rng = np.random.default_rng(21)
    lens = [13, 5, 8, 0, 17]
    interval = 4
    T, H, dk, dv = sum(lens), 2, 5, 3
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens))
    cu = np.concatenate([[0], np.cumsum(lens)])
    counts, base = oracle_mod.checkpoint_counts(cu, interval)
    assert counts.tolist() == [3, 1, 2, 0, 4]
    assert base.tolist() == [0, 3, 4, 6, 6]
    o, S, ck, _ = oracle_mod.kda_reference_checkpoints(q, k, v, z, beta, A, S0, cu,
                                                       interval=interval)
    o_ref, S_ref, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu)
    assert np.array_equal(o, o_ref) and np.array_equal(S, S_ref)
    assert ck.shape == (int(counts.sum()), H, dk, dv)
    for n in range(len(lens)):
        for m in range(1, counts[n] + 1):
            pre = slice(cu[n], cu[n] + m * interval)
            _, Sp, _ = oracle_mod.kda_reference(q[pre], k[pre], v[pre], z[pre], beta[pre], A,
                                                S0[n:n + 1])
            assert np.array_equal(ck[base[n] + m - 1], Sp[0]), (n, m)
            rest = slice(cu[n] + m * interval, cu[n + 1])
            if rest.stop > rest.start:
                orr, Srr, _ = oracle_mod.kda_reference(q[rest], k[rest], v[rest], z[rest],
                                                       beta[rest], A, ck[base[n] + m - 1][None])
                assert np.array_equal(orr, o[rest]) and np.array_equal(Srr[0], S[n])
    # length 8 = 2 intervals: the last checkpoint is the final state
    assert np.array_equal(ck[base[2] + 1], S[2])


# ------------------------------------------------- Kimi Linear softplus gate
def test_softplus_gate_closed_forms(oracle_mod):
    """g = -softplus(e^A z): g(0) = -ln 2 for any A (alpha = 1/2); alpha is the
    logistic function of -e^A z; the gate is unbounded below (about -x for
    large x) and tends to 0 for large negative arguments."""
    for A in (-1.3, 0.0, 0.7):
        assert abs(oracle_mod.gate_softplus(0.0, A) + math.log(2.0)) < 1e-15
    for z, A in ((0.3, 0.2), (-2.0, 0.5), (5.0, -0.4), (40.0, 1.0)):
        x = math.exp(A) * z
        alpha = math.exp(float(oracle_mod.gate_softplus(z, A)))
        assert abs(alpha - 1.0 / (1.0 + math.exp(x))) <= 1e-15 * max(1.0, alpha) + 1e-300
    g = float(oracle_mod.gate_softplus(1000.0, 0.0))
    assert abs(g + 1000.0) < 1e-9                  # unbounded: no -5 floor
    assert float(oracle_mod.gate_softplus(-800.0, 0.0)) > -1e-300


@pytest.mark.parametrize("T,dk,dv", [(5, 3, 2), (8, 4, 4)])
def test_softplus_gate_brute_force_products(oracle_mod, T, dk, dv):
    """The recurrence with the softplus gate equals the explicit product of the
    transition matrices (I - beta k k^T) Diag(alpha) on tiny inputs."""
    rng = np.random.default_rng(40 + T)
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, 1, dk, dv, zscale=3.0)
    o, S, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, softplus_gate=True)
    St = S0[0, 0].copy()
    for t in range(T):
        kh = _unit(k[t, 0]); qh = _unit(q[t, 0])
        x = math.exp(A[0]) * z[t, 0]
        alpha = 1.0 / (1.0 + np.exp(x))          # e^{-softplus(x)}
        St = (np.eye(dk) - beta[t, 0] * np.outer(kh, kh)) @ np.diag(alpha) @ St \
            + beta[t, 0] * np.outer(kh, v[t, 0])
        assert _close(o[t, 0], St.T @ qh, 1e-12)
    assert _close(S[0, 0], St, 1e-12)


def test_softplus_gate_chunked_equals_recurrent(oracle_mod):
    rng = np.random.default_rng(44)
    lens = [70, 3, 33]
    T, H, dk, dv = sum(lens), 2, 6, 5
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens), zscale=2.0)
    cu = np.concatenate([[0], np.cumsum(lens)])
    o_r, S_r, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu, softplus_gate=True)
    o_c, S_c, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu, chunk=16,
                                           softplus_gate=True)
    assert _close(o_c, o_r, 1e-10) and _close(S_c, S_r, 1e-10)
    o_k3, _, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0, cu)
    assert not _close(o_k3, o_r, 1e-3)             # the two gates really differ


# ------------------------------------------------ short convolution + state
# Reading of the pages' "short convolutions" / "convolution state": a causal
# depthwise convolution along time, y_t = sum_j w[:, j] x_{t-W+1+j}, whose
# state is the last W-1 inputs (oldest first).

@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_short_conv_is_numpy_convolve(oracle_mod, W):
    """With a zero state every channel is the textbook full convolution with
    the reversed taps, truncated to the sequence (numpy.convolve)."""
    rng = np.random.default_rng(60 + W)
    T, C = 11, 5
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    y, s = oracle_mod.short_conv(x, w)
    for c in range(C):
        assert _close(y[:, c], np.convolve(x[:, c], w[c, ::-1])[:T], 1e-14)
    # final state: the last W-1 inputs, oldest first
    assert np.array_equal(s[0], x[T - (W - 1):] if W > 1 else np.zeros((0, C)))


def test_short_conv_impulse_response(oracle_mod):
    """A unit impulse at t0 in one channel gives the taps in reverse order
    at t0, t0+1, ..., t0+W-1 and zero everywhere else."""
    T, C, W, t0, c0 = 9, 3, 4, 2, 1
    w = np.arange(1.0, 1.0 + C * W).reshape(C, W)
    x = np.zeros((T, C))
    x[t0, c0] = 1.0
    y, _ = oracle_mod.short_conv(x, w)
    want = np.zeros((T, C))
    for m in range(W):
        want[t0 + m, c0] = w[c0, W - 1 - m]
    assert np.array_equal(y, want)


@pytest.mark.parametrize("W", [2, 4])
def test_short_conv_state_is_prepended_input(oracle_mod, W):
    """A conv state acts as the W-1 inputs just before the sequence: running
    with state s equals running on [s; x] from a zero state and dropping the
    first W-1 outputs; the final state is the last W-1 rows of [s; x], also
    for sequences shorter than W-1."""
    rng = np.random.default_rng(70 + W)
    C = 4
    w = rng.standard_normal((C, W))
    for T in (0, 1, W - 1, 7):
        x = rng.standard_normal((T, C))
        s = rng.standard_normal((1, W - 1, C))
        y, s_out = oracle_mod.short_conv(x, w, state_in=s)
        xx = np.concatenate([s[0], x])
        yy, ss = oracle_mod.short_conv(xx, w)
        assert y.shape == (T, C) and (T == 0 or _close(y, yy[W - 1:], 1e-14))
        assert np.array_equal(s_out[0], xx[len(xx) - (W - 1):])
        assert np.array_equal(s_out, ss)


def test_short_conv_split_and_varlen(oracle_mod):
    """Packed sequences are independent (varlen = separate calls), and a
    sequence cut anywhere and resumed from the first part's conv state gives
    the same outputs and final state as one pass (prefill then decode)."""
    rng = np.random.default_rng(80)
    C, W = 6, 4
    w = rng.standard_normal((C, W))
    lens = [9, 0, 2, 13]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.standard_normal((cu[-1], C))
    s0 = rng.standard_normal((len(lens), W - 1, C))
    y, s = oracle_mod.short_conv(x, w, cu, s0, silu=True)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        yn, sn = oracle_mod.short_conv(x[sl], w, None, s0[n:n + 1], silu=True)
        assert np.array_equal(yn, y[sl]) and np.array_equal(sn[0], s[n])
    x1 = x[cu[3]:cu[4]]
    for cut in (0, 1, 2, 5, 13):
        ya, sa = oracle_mod.short_conv(x1[:cut], w, None, s0[3:4])
        parts = [ya]                 # the first part as one prefill
        st = sa
        for t in range(cut, 13):     # the rest one token at a time, as decode
            yt, st = oracle_mod.short_conv(x1[t:t + 1], w, None, st)
            parts.append(yt)
        yf, sf = oracle_mod.short_conv(x1, w, None, s0[3:4])
        assert _close(np.concatenate(parts), yf, 1e-14) and np.array_equal(st, sf)


def test_short_conv_silu_closed_forms(oracle_mod):
    """SiLU after the convolution: silu(0) = 0, silu(ln 3) = (3/4) ln 3,
    silu(-ln 3) = -(1/4) ln 3, silu(40) = 40 to rounding."""
    x = np.array([[1.0], [0.0], [0.0], [0.0]])
    for val, want in ((0.0, 0.0), (math.log(3.0), 0.75 * math.log(3.0)),
                      (-math.log(3.0), -0.25 * math.log(3.0)), (40.0, 40.0)):
        w = np.array([[0.0, val]])           # y_t = val * x_t
        y, _ = oracle_mod.short_conv(x, w, silu=True)
        assert abs(y[0, 0] - want) <= 1e-15 * max(1.0, abs(want))
        assert y[1, 0] == 0.0


@pytest.mark.parametrize("W", [1, 4])
def test_short_conv_qkv_packing(oracle_mod, W):
    """The per-head packed layouts (weights [H, 2dk+dv, W], state
    [N, H, W-1, 2dk+dv], channels q | k | v) address the same channels as
    convolving q, k and v one channel at a time."""
    rng = np.random.default_rng(90)
    T, H, dk, dv = 7, 2, 3, 2
    q, k, v = (rng.standard_normal((T, H, d)) for d in (dk, dk, dv))
    cw = rng.standard_normal((H, 2 * dk + dv, W))
    st = rng.standard_normal((1, H, W - 1, 2 * dk + dv))
    qc, kc, vc, so = oracle_mod.short_conv_qkv(q, k, v, cw, None, st)
    for h in range(H):
        for name, xin, out, off, d in (("q", q, qc, 0, dk), ("k", k, kc, dk, dk),
                                       ("v", v, vc, 2 * dk, dv)):
            for c in range(d):
                xs = np.concatenate([st[0, h, :, off + c], xin[:, h, c]])
                want = np.convolve(xs, cw[h, off + c, ::-1])[W - 1:W - 1 + T]
                assert _close(out[:, h, c], want, 1e-14), name
                assert np.array_equal(so[0, h, :, off + c], xs[len(xs) - (W - 1):])


def test_conv_kda_prefill_equals_decode_steps(oracle_mod):
    """Convolution + KDA over a sequence equals the same sequence fed one
    token at a time with both states (recurrent and conv) carried between
    steps: the decode loop with persistent states."""
    rng = np.random.default_rng(95)
    T, H, dk, dv, W = 6, 2, 4, 3, 4
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    cw = 0.5 * rng.standard_normal((H, 2 * dk + dv, W))
    cs0 = rng.standard_normal((1, H, W - 1, 2 * dk + dv))
    o, S, cs = oracle_mod.kda_reference_conv(q, k, v, z, beta, A, cw, cs0, S0, silu=True)
    St, ct = S0, cs0
    for t in range(T):
        sl = slice(t, t + 1)
        ot, St, ct = oracle_mod.kda_reference_conv(q[sl], k[sl], v[sl], z[sl], beta[sl], A,
                                                   cw, ct, St, silu=True)
        assert _close(ot, o[sl], 1e-12)
    assert _close(St, S, 1e-12) and np.array_equal(ct, cs)
    # and the convolution really acts: without it the output differs
    o_plain, _, _ = oracle_mod.kda_reference(q, k, v, z, beta, A, S0)
    assert not _close(o_plain, o, 1e-3)


# ------------------------------------------- reverse mode (training backward)
def _loss(oracle_mod, dO, dSf, cu, flags, **x):
    o, S, _ = oracle_mod.kda_reference(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                                       x["S0"], cu, **flags)
    return float((o * dO).sum() + (0.0 if dSf is None else (S * dSf).sum()))


@pytest.mark.parametrize("softplus,l2norm,with_state", [(False, True, True), (True, True, False),
                                                        (False, False, True)])
def test_backward_matches_finite_differences(oracle_mod, softplus, l2norm, with_state):
    """Directional derivatives of L = sum(dO * o) + sum(dSf * S_T), taken by
    central differences of the forward oracle (step 1e-6 in fp64), equal the
    reverse-mode gradients contracted with the same directions, for every
    input; varlen with an empty sequence."""
    rng = np.random.default_rng(500 + 2 * softplus + l2norm)
    lens = [5, 0, 3]
    T, H, dk, dv = sum(lens), 2, 4, 3
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens), zscale=2.0)
    if not with_state:
        S0 = None
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lens), H, dk, dv)) if with_state else None
    flags = dict(softplus_gate=softplus, l2norm=l2norm, scale=0.7)
    g = oracle_mod.kda_reference_backward(q, k, v, z, beta, A, S0, cu, dO, dSf, **flags)
    x = dict(q=q, k=k, v=v, z=z, beta=beta, A=A, S0=S0)
    keys = dict(q="dq", k="dk", v="dv", z="dz", beta="dbeta", A="dA", S0="dS0")
    eps = 1e-6
    for name, key in keys.items():
        if x[name] is None:
            continue
        d = rng.standard_normal(x[name].shape)
        xp, xm = dict(x), dict(x)
        xp[name] = x[name] + eps * d
        xm[name] = x[name] - eps * d
        fd = (_loss(oracle_mod, dO, dSf, cu, flags, **xp) -
              _loss(oracle_mod, dO, dSf, cu, flags, **xm)) / (2 * eps)
        an = float((g[key] * d).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_backward_matches_autograd(oracle_mod):
    """The reverse-mode gradients equal torch.autograd of a separate fp64
    torch restatement of the recurrence (gate, normalisation, delta rule,
    read after write) on one sequence."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(510)
    T, H, dk, dv = 6, 2, 5, 4
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv)
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((1, H, dk, dv))
    g = oracle_mod.kda_reference_backward(q, k, v, z, beta, A, S0, None, dO, dSf, scale=1.3)
    tt = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True)
          for n, a in dict(q=q, k=k, v=v, z=z, beta=beta, A=A, S0=S0).items()}
    L = 0.0
    for h in range(H):
        S = tt["S0"][0, h]
        for t in range(T):
            qh = 1.3 * tt["q"][t, h] / torch.sqrt((tt["q"][t, h] ** 2).sum() + 1e-6)
            kh = tt["k"][t, h] / torch.sqrt((tt["k"][t, h] ** 2).sum() + 1e-6)
            alpha = torch.exp(-5.0 * torch.sigmoid(torch.exp(tt["A"][h]) * tt["z"][t, h]))
            b = tt["beta"][t, h]
            Sd = alpha[:, None] * S
            S = Sd - b * torch.outer(kh, kh @ Sd) + b * torch.outer(kh, tt["v"][t, h])
            L = L + (S.T @ qh * torch.tensor(dO[t, h])).sum()
        L = L + (S * torch.tensor(dSf[0, h])).sum()
    L.backward()
    for n, key in dict(q="dq", k="dk", v="dv", z="dz", beta="dbeta", A="dA", S0="dS0").items():
        assert _close(g[key], tt[n].grad.numpy(), 1e-10), n


def test_backward_identity_closed_form(oracle_mod):
    """alpha = 1 (saturated gate), beta = 0: o_t = S0^T qh_t and S_T = S0, so
    dS0 = sum_t qh_t dO_t^T + dSf, dv = 0, dz = 0, dA = 0, and dqh_t = S0 dO_t
    (no normalisation here, scale 1)."""
    rng = np.random.default_rng(520)
    T, H, dk, dv = 4, 1, 3, 2
    q, k, v, _, _, _, S0 = _rand_case(rng, T, H, dk, dv)
    z = np.full((T, H, dk), -1e4)
    A = np.zeros(H)
    beta = np.zeros((T, H))
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((1, H, dk, dv))
    g = oracle_mod.kda_reference_backward(q, k, v, z, beta, A, S0, None, dO, dSf, l2norm=False)
    want = dSf[0, 0] + sum(np.outer(q[t, 0], dO[t, 0]) for t in range(T))
    assert _close(g["dS0"][0, 0], want, 1e-13)
    assert np.all(g["dv"] == 0.0) and np.all(g["dz"] == 0.0) and g["dA"][0] == 0.0
    for t in range(T):
        assert _close(g["dq"][t, 0], S0[0, 0] @ dO[t, 0], 1e-13)


@pytest.mark.parametrize("softplus,l2norm", [(False, True), (True, True), (False, False)])
@pytest.mark.parametrize("C", [1, 3, 16, 64])
def test_backward_chunked_form_equals_reverse_mode(oracle_mod, softplus, l2norm, C):
    """The chunked form of the backward (in-chunk cumulative gate, UT system
    and its transpose, chunks walked last to first with dL/dS carried between
    them) gives the reverse-mode gradients of the recurrence for every input:
    chunk sizes that do and do not divide the lengths, an empty sequence, a
    sequence shorter than one chunk, nonzero S0 and dL/dS_T, scale != 1."""
    rng = np.random.default_rng(530 + C + 2 * softplus + l2norm)
    lens = [70, 0, 5, 33]
    T, H, dk, dv = sum(lens), 2, 6, 5
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, z, beta, A, S0 = _rand_case(rng, T, H, dk, dv, N=len(lens), zscale=2.0)
    dO = rng.standard_normal((T, H, dv))
    dSf = rng.standard_normal((len(lens), H, dk, dv))
    flags = dict(softplus_gate=softplus, l2norm=l2norm, scale=0.8)
    ref = oracle_mod.kda_reference_backward(q, k, v, z, beta, A, S0, cu, dO, dSf, **flags)
    got = oracle_mod.kda_reference_backward_chunked(q, k, v, z, beta, A, S0, cu, dO, dSf,
                                                    chunk=C, **flags)
    for key in ("dq", "dk", "dv", "dz", "dbeta", "dA", "dS0"):
        assert _close(got[key], ref[key], 1e-10), key
