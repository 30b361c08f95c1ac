"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test states which fact it checks and which part of the method it
guards.  Pins use: exact rational arithmetic (fractions) on tiny inputs,
closed forms for the beta = 0 and decay = 1 special cases, the delta-rule
fixed point, the gate's special values (sigmoid(0) = 1/2, softplus(0) = ln 2,
saturation), and structural identities (split/chain, varlen packing).  K != V
throughout where a transposed state would otherwise go unnoticed.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def _rand(*shape, std=1.0):
    return (RNG.standard_normal(shape) * std).astype(np.float32)


# ---------------------------------------------------------------------------
# Gate special values (fla-kda SKILL.md, "Gate contracts")
# ---------------------------------------------------------------------------

def test_gate_special_values_numpy():
    lb = -3.0
    # sigmoid(0) = 1/2  -> safe gate = lb/2 at z = 0 for any A_log
    assert oracle.gate_activation(0.0, 0.7, "safe", lb) == lb / 2
    # saturation: z -> +inf gives lb, z -> -inf gives 0 (exactly, in fp64)
    assert oracle.gate_activation(1e4, 0.0, "safe", lb) == lb
    assert oracle.gate_activation(-1e4, 0.0, "safe", lb) == 0.0
    # A_log omitted -> multiplier one: sigmoid(1) for z = 1
    assert math.isclose(oracle.gate_activation(1.0, None, "safe", lb), lb / (1 + math.exp(-1)),
                        rel_tol=1e-15)
    # softplus(0) = ln 2  -> unsafe gate = -exp(A_log) ln 2
    assert math.isclose(oracle.gate_activation(0.0, 0.0, "unsafe", lb), -math.log(2), rel_tol=1e-15)
    assert math.isclose(oracle.gate_activation(0.0, math.log(3.0), "unsafe", lb),
                        -3 * math.log(2), rel_tol=1e-14)
    # softplus(z) -> z for large z, -> e^z for very negative z
    assert math.isclose(oracle.gate_activation(50.0, 0.0, "unsafe", lb), -50.0, rel_tol=1e-15)
    assert math.isclose(oracle.gate_activation(-30.0, 0.0, "unsafe", lb), -math.exp(-30.0),
                        rel_tol=1e-12)
    assert oracle.gate_activation(-1e4, 0.0, "unsafe", lb) == 0.0


def test_safe_gate_range_invariant():
    """I7: every safe log-decay lies in [lower_bound, 0]."""
    z = np.concatenate([RNG.standard_normal(10000) * 30, [1e4, -1e4, 0.0, 88.0, -88.0]])
    for lb in (-5.0, -1e-3, -2.5):
        for A_log in (None, -4.6, 0.0, 4.1):
            a = oracle.gate_activation(z, A_log, "safe", lb)
            assert np.all(a <= 0.0) and np.all(a >= lb)


def _decay_via_recurrence(gvals, gate, lb, A_log):
    """Recover exp(a_t) from the C oracle with K = V = 1, beta = 0, S0 = 1,
    q = 1: then o_t = scale * prod_{s<=t} exp(a_s)."""
    T = len(gvals)
    one = np.ones((1, T, 1, 1), np.float32)
    g = np.asarray(gvals, np.float32).reshape(1, T, 1, 1)
    beta = np.full((1, T, 1), -1e4, np.float32)
    init = np.ones((1, 1, 1, 1), np.float32)
    out, fin = oracle.kda_recurrence(one, one, one, g, beta, scale=1.0, gate=gate, lower_bound=lb,
                                     A_log=None if A_log is None else np.float32([A_log]),
                                     initial_state=init)
    o = out.reshape(T)
    return np.concatenate([[o[0]], o[1:] / o[:-1]]), fin.reshape(())


def test_gate_through_c_recurrence():
    """The C oracle's own gate: decay exactly 1/2 for z = 0 with lb = -2 ln 2
    (safe) or A_log = 0 (unsafe); decay 1 for saturated negative logits; the
    safe decay floor exp(lb) for saturated positive logits."""
    lb = -2 * math.log(2)
    d, _ = _decay_via_recurrence([0.0, -1e4, 1e4, 0.0], "safe", lb, 0.3)
    np.testing.assert_allclose(d, [0.5, 1.0, math.exp(lb), 0.5], rtol=1e-14)
    d, _ = _decay_via_recurrence([0.0, -1e4, 0.0], "unsafe", -5.0, 0.0)
    np.testing.assert_allclose(d, [0.5, 1.0, 0.5], rtol=1e-14)
    d, _ = _decay_via_recurrence([0.0], "unsafe", -5.0, math.log(3.0))
    np.testing.assert_allclose(d, [0.125], rtol=1e-6)  # A_log stored in fp32
    # A_log omitted in safe mode -> multiplier one
    d, _ = _decay_via_recurrence([1.0], "safe", -1.0, None)
    np.testing.assert_allclose(d, [math.exp(-1.0 / (1 + math.exp(-1.0)))], rtol=1e-14)


# ---------------------------------------------------------------------------
# Exact rational recurrence on tiny inputs (brute force, fractions)
# ---------------------------------------------------------------------------

def _exact_recurrence(q, k, v, decay, beta, S0, scale):
    """Brute force in exact rationals: S <- S Diag(decay_t); S <- S + beta_t
    (v_t - S k_t) k_t^T; o_t = scale S q_t.  Lists of Fractions."""
    V, K = len(S0), len(S0[0])
    S = [row[:] for row in S0]
    outs = []
    for t in range(len(q)):
        S = [[S[r][c] * decay[t][c] for c in range(K)] for r in range(V)]
        pred = [sum(S[r][c] * k[t][c] for c in range(K)) for r in range(V)]
        S = [[S[r][c] + beta[t] * (v[t][r] - pred[r]) * k[t][c] for c in range(K)]
             for r in range(V)]
        outs.append([scale * sum(S[r][c] * q[t][c] for c in range(K)) for r in range(V)])
    return outs, S


@pytest.mark.parametrize("gate", ["safe", "unsafe"])
def test_exact_rational_example(gate):
    """K = 2, V = 3, T = 4.  Channel 0 decays by exactly 1/2 per token
    (z = 0: sigmoid(0) = 1/2 with lb = -2 ln 2, or softplus(0) = ln 2 with
    A_log = 0), channel 1 by exactly 1 (z = -1e4 saturates the gate to 0).
    beta logits 0 give beta = 1/2.  The expected values are exact rationals."""
    T, K, V = 4, 2, 3
    F = Fraction
    qv = [[F(1), F(-1, 2)], [F(1, 4), F(3, 4)], [F(-1), F(1, 2)], [F(3, 8), F(1)]]
    kv = [[F(1, 2), F(1)], [F(-1, 4), F(1, 2)], [F(1), F(1, 4)], [F(1, 2), F(-1, 2)]]
    vv = [[F(1), F(2), F(-1)], [F(0), F(1, 2), F(1)], [F(-3, 2), F(1), F(1, 4)],
          [F(2), F(-1), F(1, 2)]]
    S0 = [[F(1, 4), F(-1, 2)], [F(1), F(1, 8)], [F(-1, 2), F(3, 4)]]
    decay = [[F(1, 2), F(1)]] * T
    beta = [F(1, 2)] * T
    scale = F(1, 2)
    eo, eS = _exact_recurrence(qv, kv, vv, decay, beta, S0, scale)

    f32 = lambda rows: np.array([[float(x) for x in r] for r in rows], np.float32)
    q = f32(qv).reshape(1, T, 1, K)
    k = f32(kv).reshape(1, T, 1, K)
    v = f32(vv).reshape(1, T, 1, V)
    g = np.tile(np.float32([0.0, -1e4]), (T, 1)).reshape(1, T, 1, K)
    b = np.zeros((1, T, 1), np.float32)
    init = f32(S0).reshape(1, 1, V, K)
    lb = -2 * math.log(2) if gate == "safe" else -5.0
    kw = dict(scale=0.5, gate=gate, lower_bound=lb, A_log=np.float32([0.0]), initial_state=init)
    out, fin = oracle.kda_recurrence(q, k, v, g, b, **kw)
    np.testing.assert_allclose(out.reshape(T, V), np.array(eo, dtype=np.float64), rtol=1e-14,
                               atol=1e-15)
    np.testing.assert_allclose(fin.reshape(V, K), np.array(eS, dtype=np.float64), rtol=1e-14,
                               atol=1e-15)
    out2, fin2 = oracle.chunk_form(q, k, v, g, b, chunk=2, **kw)
    np.testing.assert_allclose(out2.reshape(T, V), np.array(eo, dtype=np.float64), rtol=1e-13,
                               atol=1e-14)
    np.testing.assert_allclose(fin2.reshape(V, K), np.array(eS, dtype=np.float64), rtol=1e-13,
                               atol=1e-14)


# ---------------------------------------------------------------------------
# I1: brute force as a product of affine maps (numpy matrices), K != V
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,V,T", [(2, 2, 3), (3, 2, 4), (2, 3, 4), (3, 3, 1)])
@pytest.mark.parametrize("gate", ["safe", "unsafe"])
def test_affine_map_brute_force(K, V, T, gate):
    """S_t = S_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, composed
    with a generic matrix routine; outputs o_t = scale S_t q_t."""
    q, k, g = _rand(1, T, 1, K), _rand(1, T, 1, K), _rand(1, T, 1, K)
    v, b = _rand(1, T, 1, V), _rand(1, T, 1)
    A_log, dtb, init = np.float32([0.4]), _rand(1, K, std=0.1), _rand(1, 1, V, K)
    kw = dict(scale=0.7, gate=gate, lower_bound=-4.0, A_log=A_log, dt_bias=dtb, initial_state=init)
    out, fin = oracle.kda_recurrence(q, k, v, g, b, **kw)
    S = init[0, 0].astype(np.float64)
    for t in range(T):
        a = oracle.gate_activation(g[0, t, 0].astype(np.float64) + dtb[0], A_log[0], gate, -4.0)
        bt = 1.0 / (1.0 + np.exp(-np.float64(b[0, t, 0])))
        kt = k[0, t, 0].astype(np.float64)
        M = np.diag(np.exp(a)) @ (np.eye(K) - bt * np.outer(kt, kt))
        S = S @ M + bt * np.outer(v[0, t, 0].astype(np.float64), kt)
        np.testing.assert_allclose(out[0, t, 0], 0.7 * S @ q[0, t, 0].astype(np.float64),
                                   rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("K,V,T", [(3, 2, 4), (2, 3, 3)])
def test_affine_map_brute_force_modes(K, V, T):
    """The same brute force for the caller-gated mode (g is the log decay a_t
    itself; dt_bias and A_log are given but must not be used) with beta given
    as beta itself (no sigmoid)."""
    q, k = _rand(1, T, 1, K), _rand(1, T, 1, K)
    a_in = (-np.abs(_rand(1, T, 1, K))).astype(np.float32)  # log decays <= 0
    v = _rand(1, T, 1, V)
    b = np.float32(np.random.default_rng(7).uniform(0.05, 0.95, (1, T, 1)))
    A_log, dtb, init = np.float32([0.4]), _rand(1, K, std=0.5), _rand(1, 1, V, K)
    kw = dict(scale=0.7, gate="logspace", beta_prob=True, A_log=A_log, dt_bias=dtb,
              initial_state=init)
    out, fin = oracle.kda_recurrence(q, k, v, a_in, b, **kw)
    S = init[0, 0].astype(np.float64)
    for t in range(T):
        bt = np.float64(b[0, t, 0])
        kt = k[0, t, 0].astype(np.float64)
        M = np.diag(np.exp(a_in[0, t, 0].astype(np.float64))) @ (np.eye(K) - bt * np.outer(kt, kt))
        S = S @ M + bt * np.outer(v[0, t, 0].astype(np.float64), kt)
        np.testing.assert_allclose(out[0, t, 0], 0.7 * S @ q[0, t, 0].astype(np.float64),
                                   rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-13, atol=1e-13)
    out2, fin2 = oracle.chunk_form(q, k, v, a_in, b, chunk=2, **kw)
    np.testing.assert_allclose(out2, out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fin2, fin, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# I2: beta = 0 -> diagonal-gated linear read-out, closed form
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gate", ["safe", "unsafe"])
def test_beta_zero_closed_form(gate):
    T, H, K, V = 37, 2, 5, 3
    q, k, g, v = _rand(1, T, H, K), _rand(1, T, H, K), _rand(1, T, H, K), _rand(1, T, H, V)
    b = np.full((1, T, H), -1e4, np.float32)  # sigmoid(-1e4) == 0 exactly in fp64
    A_log, dtb, init = _rand(H, std=0.5), _rand(H, K, std=0.1), _rand(1, H, V, K)
    kw = dict(scale=0.3, gate=gate, lower_bound=-2.0, A_log=A_log, dt_bias=dtb, initial_state=init)
    out, fin = oracle.kda_recurrence(q, k, v, g, b, **kw)
    for h in range(H):
        a = oracle.gate_activation(g[0, :, h].astype(np.float64) + dtb[h], A_log[h], gate, -2.0)
        Gam = np.cumsum(a, axis=0)
        S0 = init[0, h].astype(np.float64)
        expect = 0.3 * (np.exp(Gam) * q[0, :, h]) @ S0.T
        np.testing.assert_allclose(out[0, :, h], expect, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fin[0, h], S0 * np.exp(Gam[-1])[None, :], rtol=1e-12,
                                   atol=1e-14)


# ---------------------------------------------------------------------------
# I3: decay exactly 1 with distinct one-hot keys, closed form
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gate", ["safe", "unsafe"])
def test_unit_decay_one_hot_keys(gate):
    T, K, V = 6, 8, 5
    idx = RNG.permutation(K)[:T]
    k = np.zeros((1, T, 1, K), np.float32)
    k[0, np.arange(T), 0, idx] = 1.0
    q, v = _rand(1, T, 1, K), _rand(1, T, 1, V)
    g = np.full((1, T, 1, K), -1e4, np.float32)  # gate saturates to a = 0 in both modes
    b = _rand(1, T, 1)
    init = _rand(1, 1, V, K)
    kw = dict(scale=1.0, gate=gate, lower_bound=-5.0, A_log=np.float32([0.2]), initial_state=init)
    out, fin = oracle.kda_recurrence(q, k, v, g, b, **kw)
    S = init[0, 0].astype(np.float64).copy()
    S0 = S.copy()
    for t in range(T):
        bt = 1.0 / (1.0 + np.exp(-np.float64(b[0, t, 0])))
        S[:, idx[t]] = S0[:, idx[t]] + bt * (v[0, t, 0] - S0[:, idx[t]])
        np.testing.assert_allclose(out[0, t, 0], S @ q[0, t, 0], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-13, atol=1e-14)
    # and with beta = 0 as well the read-out is plain linear attention on S0
    b0 = np.full_like(b, -1e4)
    out0, _ = oracle.kda_recurrence(q, k, v, g, b0, **kw)
    np.testing.assert_allclose(out0[0, :, 0], q[0, :, 0] @ S0.T, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# I4: delta-rule fixed point with L2 norm and beta = 1; L2-norm invariance
# ---------------------------------------------------------------------------

def test_delta_rule_fixed_point():
    T, K, V = 5, 6, 4
    q, k, g, v = _rand(1, T, 1, K), _rand(1, T, 1, K), _rand(1, T, 1, K), _rand(1, T, 1, V)
    b = np.full((1, T, 1), 40.0, np.float32)  # sigmoid(40) rounds to 1.0 in fp64
    kw = dict(scale=1.0, gate="safe", lower_bound=-1.0, A_log=np.float32([0.0]), qk_l2norm=True,
              initial_state=_rand(1, 1, V, K))
    for t in range(1, T + 1):
        _, fin = oracle.kda_recurrence(q[:, :t], k[:, :t], v[:, :t], g[:, :t], b[:, :t], **kw)
        kt = k[0, t - 1, 0].astype(np.float64)
        khat = kt / np.sqrt(kt @ kt + 1e-6)
        np.testing.assert_allclose(fin[0, 0] @ khat, v[0, t - 1, 0], rtol=1e-6, atol=1e-6)


def test_l2norm_scale_invariance():
    """With in-kernel L2 norm, rescaling q and k by positive factors changes
    nothing (up to the epsilon), and without it the output is linear in q."""
    T, H, K, V = 20, 1, 16, 8
    q, k, g, v, b = (_rand(1, T, H, K), _rand(1, T, H, K), _rand(1, T, H, K), _rand(1, T, H, V),
                     _rand(1, T, H))
    kw = dict(scale=0.5, gate="safe", lower_bound=-3.0, A_log=np.float32([0.1]), qk_l2norm=True)
    o1, f1 = oracle.kda_recurrence(q, k, v, g, b, **kw)
    s = np.float32(8.0)
    o2, f2 = oracle.kda_recurrence(q * s, k * np.float32(0.25) * s, v, g, b, **kw)
    np.testing.assert_allclose(o2, o1, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(f2, f1, rtol=1e-6, atol=1e-7)
    kw["qk_l2norm"] = False
    o3, _ = oracle.kda_recurrence(q, k, v, g, b, **kw)
    o4, _ = oracle.kda_recurrence(q * np.float32(2.0), k, v, g, b, **kw)
    np.testing.assert_allclose(o4, 2 * o3, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# I5 / I6: split-and-chain, varlen packing
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("split", [16, 64, 37, 1])
def test_split_chain(split):
    T, H, K, V = 130, 2, 8, 6
    args = [_rand(1, T, H, K), _rand(1, T, H, K), _rand(1, T, H, V), _rand(1, T, H, K),
            _rand(1, T, H)]
    kw = dict(scale=0.2, gate="unsafe", A_log=_rand(H, std=0.3), dt_bias=_rand(H, K, std=0.1),
              qk_l2norm=True)
    init = _rand(1, H, V, K)
    o_full, f_full = oracle.kda_recurrence(*args, initial_state=init, **kw)
    a1 = [x[:, :split] for x in args]
    a2 = [x[:, split:] for x in args]
    o1, f1 = oracle.kda_recurrence(*a1, initial_state=init, **kw)
    o2, f2 = oracle.kda_recurrence(*a2, initial_state=f1.astype(np.float32), **kw)
    # the intermediate state is rounded to fp32 when handed over: compare loosely
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o_full, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(f2, f_full, rtol=1e-5, atol=1e-6)
    np.testing.assert_array_equal(o1, o_full[:, :split])  # prefix identical


def test_varlen_pack_equals_separate():
    lens = [5, 1, 64, 17, 33]
    H, K, V = 2, 8, 4
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    Tt = int(cu[-1])
    args = [_rand(1, Tt, H, K), _rand(1, Tt, H, K), _rand(1, Tt, H, V), _rand(1, Tt, H, K),
            _rand(1, Tt, H)]
    init = _rand(len(lens), H, V, K)
    kw = dict(scale=0.4, gate="safe", lower_bound=-5.0, A_log=_rand(H), dt_bias=_rand(H, K),
              qk_l2norm=True)
    o, f = oracle.kda_recurrence(*args, cu_seqlens=cu, initial_state=init, **kw)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        on, fn = oracle.kda_recurrence(*[x[:, sl] for x in args], initial_state=init[n:n + 1], **kw)
        np.testing.assert_array_equal(o[:, sl], on)
        np.testing.assert_array_equal(f[n], fn[0])


def test_units_subset_matches_full():
    T, H, K, V = 40, 3, 8, 8
    args = [_rand(2, T, H, K), _rand(2, T, H, K), _rand(2, T, H, V), _rand(2, T, H, K),
            _rand(2, T, H)]
    kw = dict(scale=0.4, gate="safe", lower_bound=-5.0, A_log=_rand(H))
    o, f = oracle.kda_recurrence(*args, **kw)
    o2, f2 = oracle.kda_recurrence(*args, units=[4, 1], **kw)  # (n=1,h=1), (n=0,h=1)
    np.testing.assert_array_equal(o2[1, :, 1], o[1, :, 1])
    np.testing.assert_array_equal(o2[0, :, 1], o[0, :, 1])
    assert np.isnan(o2[0, :, 0]).all()
    np.testing.assert_array_equal(f2[1, 1], f[1, 1])


# ---------------------------------------------------------------------------
# Chunk form against the recurrence (two independent restatements)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gate,l2,chunk,with_init", [("safe", True, 16, True),
                                                     ("unsafe", True, 16, False),
                                                     ("safe", False, 64, True),
                                                     ("unsafe", False, 8, True)])
def test_chunk_form_matches_recurrence(gate, l2, chunk, with_init):
    B, T, H, K, V = 2, 75, 2, 16, 12
    args = [_rand(B, T, H, K), _rand(B, T, H, K), _rand(B, T, H, V), _rand(B, T, H, K),
            _rand(B, T, H)]
    kw = dict(scale=0.25, gate=gate, lower_bound=-5.0, A_log=_rand(H, std=0.5),
              dt_bias=_rand(H, K, std=0.1), qk_l2norm=l2,
              initial_state=_rand(B, H, V, K) if with_init else None)
    o, f = oracle.kda_recurrence(*args, **kw)
    o2, f2 = oracle.chunk_form(*args, chunk=chunk, **kw)
    np.testing.assert_allclose(o2, o, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(f2, f, rtol=1e-10, atol=1e-11)


def test_chunk_form_varlen_and_intermediates():
    lens = [70, 3, 64]
    H, K, V = 1, 8, 8
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    Tt = int(cu[-1])
    args = [_rand(1, Tt, H, K), _rand(1, Tt, H, K), _rand(1, Tt, H, V), _rand(1, Tt, H, K),
            _rand(1, Tt, H)]
    kw = dict(scale=0.25, gate="safe", lower_bound=-5.0, A_log=_rand(H), qk_l2norm=True,
              cu_seqlens=cu)
    o, f = oracle.kda_recurrence(*args, **kw)
    o2, f2, kept = oracle.chunk_form(*args, chunk=16, keep=True, **kw)
    np.testing.assert_allclose(o2, o, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(f2, f, rtol=1e-10, atol=1e-11)
    # T is (I + A)^-1 Diag(beta): (I + A) T == Diag(beta), A strictly lower
    for ch in kept[(0, 0)]:
        L = ch["A"].shape[0]
        np.testing.assert_allclose((np.eye(L) + ch["A"]) @ ch["T"], np.diag(ch["beta"]),
                                   atol=1e-12)
        assert np.all(np.triu(ch["A"]) == 0)
    assert len(kept[(0, 0)]) == 5 and len(kept[(1, 0)]) == 1 and len(kept[(2, 0)]) == 4
