"""Pins of the fp64 backward oracle (oracle/backward.py), no GPU.

* Its forward equals the C token-recurrence oracle (itself pinned in
  test_oracle_pins.py) for every gate form, both beta modes, with and without
  the L2 norm, states and packed sequences.
* Its gradients equal central finite differences of the C oracle's loss on
  tiny inputs (every input tensor, every element): so a wrong derivative and a
  wrong forward both fail.
* Special cases: beta = 0 leaves the loss independent of v and k (exact zero
  gradients); the gradient of the final state with respect to the initial
  state is the product of the per-token transitions (brute force with the
  affine maps, K != V).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(B=1, T=5, H=2, K=4, V=3, seed=0, states=True, lengths=None):
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int64)
        B, T = 1, int(cu[-1])
    N = len(lengths) if lengths is not None else B
    r = lambda *s, sd=1.0: torch.randn(s, generator=gen, dtype=torch.float64) * sd
    return dict(q=r(B, T, H, K), k=r(B, T, H, K, sd=0.5), v=r(B, T, H, V), g=r(B, T, H, K),
                beta=r(B, T, H), A_log=torch.log(1 + 3 * torch.rand(H, generator=gen, dtype=torch.float64)),
                dt_bias=r(H, K, sd=0.1), initial_state=r(N, H, V, K, sd=0.3) if states else None,
                cu_seqlens=cu, N=N)


MODES = [dict(gate="safe", lower_bound=-5.0, qk_l2norm=True, beta_prob=False),
         dict(gate="safe", lower_bound=-0.7, qk_l2norm=False, beta_prob=False),
         dict(gate="unsafe", lower_bound=0.0, qk_l2norm=True, beta_prob=False),
         dict(gate="logspace", lower_bound=0.0, qk_l2norm=False, beta_prob=True)]


def _prep(inp, mode):
    inp = dict(inp)
    if mode["gate"] == "logspace":
        inp["g"] = -inp["g"].abs()
    if mode["beta_prob"]:
        inp["beta"] = torch.sigmoid(inp["beta"])
    return inp


@pytest.mark.parametrize("mode", MODES, ids=[m["gate"] + ("_l2" if m["qk_l2norm"] else "") for m in MODES])
def test_torch_forward_equals_c_oracle(mode):
    """The autograd forward is the C oracle's recurrence (K = V = 128 packed
    sequences with states and a dense batch)."""
    for kw in (dict(B=1, T=0, H=2, K=128, V=128, lengths=[3, 0, 17], seed=1),
               dict(B=2, T=9, H=2, K=128, V=128, seed=2)):
        inp = _prep(_inputs(**kw), mode)
        o_t, f_t = oracle.kda_forward_torch(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                            scale=0.1, A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                                            initial_state=inp["initial_state"],
                                            cu_seqlens=inp["cu_seqlens"], **mode)
        o_c, f_c = oracle.kda_recurrence(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=0.1,
                                         A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                                         initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                                         **mode)
        # the C oracle reads its inputs in fp32: compare on fp32-exact inputs
        assert np.abs(o_t.detach().numpy() - o_c).max() < 1e-5 * max(1.0, np.abs(o_c).max())
        assert np.abs(f_t.detach().numpy() - f_c).max() < 1e-5 * max(1.0, np.abs(f_c).max())


def _fp32_exact(inp):
    return {k: (v.float().double() if torch.is_tensor(v) and v.is_floating_point() else v)
            for k, v in inp.items()}


@pytest.mark.parametrize("mode", MODES, ids=[m["gate"] + ("_l2" if m["qk_l2norm"] else "") for m in MODES])
def test_torch_forward_equals_c_oracle_exact_inputs(mode):
    """Same, on inputs that fp32 holds exactly: agreement to fp64 rounding."""
    inp = _fp32_exact(_prep(_inputs(B=1, T=0, H=2, K=128, V=128, lengths=[5, 1, 12], seed=3), mode))
    o_t, f_t = oracle.kda_forward_torch(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=0.1,
                                        A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                                        initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"],
                                        **mode)
    o_c, f_c = oracle.kda_recurrence(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=0.1,
                                     A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                                     initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"], **mode)
    np.testing.assert_allclose(o_t.detach().numpy(), o_c, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(f_t.detach().numpy(), f_c, rtol=1e-10, atol=1e-12)


def _loss_c(inp, mode, dout, dfinal):
    o, f = oracle.kda_recurrence(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=0.3,
                                 A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                                 initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"], **mode)
    return float((o * dout).sum() + (f * dfinal).sum())


@pytest.mark.parametrize("mode", MODES, ids=[m["gate"] + ("_l2" if m["qk_l2norm"] else "") for m in MODES])
@pytest.mark.parametrize("packed", [False, True])
def test_gradients_equal_finite_differences(mode, packed):
    """Every element of every input's gradient against a central difference of
    the C oracle's loss (K = V = 128 would be slow; the C oracle and the torch
    forward both take any K, V, so K = 4, V = 3)."""
    kw = dict(H=2, K=4, V=3, seed=7, lengths=[3, 4]) if packed else dict(B=2, T=4, H=2, K=4, V=3, seed=8)
    inp = _fp32_exact(_prep(_inputs(**kw), mode))
    gen = torch.Generator().manual_seed(9)
    B, T, H, V = inp["v"].shape
    dout = torch.randn((B, T, H, V), generator=gen, dtype=torch.float64).float().double().numpy()
    dfinal = torch.randn(inp["initial_state"].shape, generator=gen, dtype=torch.float64).float().double().numpy()
    gr = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, scale=0.3,
                             A_log=inp["A_log"], dt_bias=inp["dt_bias"], initial_state=inp["initial_state"],
                             dfinal=dfinal, cu_seqlens=inp["cu_seqlens"], **mode)
    names = ["q", "k", "v", "g", "beta", "initial_state"]
    if mode["gate"] != "logspace":
        names += ["A_log", "dt_bias"]
    eps = 2.0 ** -16  # a power of two: x +- eps is exact in fp32 for these magnitudes
    for name in names:
        x = inp[name]
        fd = np.zeros(tuple(x.shape))
        for idx in np.ndindex(*x.shape):
            plus, minus = dict(inp), dict(inp)
            xp, xm = x.clone(), x.clone()
            xp[idx] += eps
            xm[idx] -= eps
            plus[name], minus[name] = xp, xm
            fd[idx] = (_loss_c(plus, mode, dout, dfinal) - _loss_c(minus, mode, dout, dfinal)) / (2 * eps)
        ad = gr[name]
        err = np.abs(ad - fd).max()
        assert err <= 2e-6 * max(1.0, np.abs(fd).max()), (name, err, np.abs(fd).max())


def test_beta_zero_gives_no_gradient_to_v_and_k():
    """beta = 0 (beta given as beta): no write ever happens, so the loss does
    not depend on v or k; with the L2 norm off, k is unused too."""
    mode = dict(gate="safe", lower_bound=-5.0, qk_l2norm=False, beta_prob=True)
    inp = _inputs(B=1, T=6, H=2, K=4, V=3, seed=11)
    inp["beta"] = torch.zeros_like(inp["beta"])
    dout = np.ones((1, 6, 2, 3))
    gr = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, scale=0.5,
                             A_log=inp["A_log"], dt_bias=inp["dt_bias"], initial_state=inp["initial_state"],
                             **mode)
    assert np.all(gr["v"] == 0) and np.all(gr["k"] == 0)
    assert np.abs(gr["q"]).max() > 0 and np.abs(gr["g"]).max() > 0


def test_initial_state_gradient_is_the_transition_product():
    """With dout = 0 and dfinal = E (one-hot), dL/dS0 = E (prod_t J_t)^T where
    J_t = Diag(d_t) (I - beta_t k_t k_t^T) is the per-token map of S (row
    vector form): brute force with explicit K x K matrices, K = 4 != V = 3."""
    mode = dict(gate="unsafe", lower_bound=0.0, qk_l2norm=True, beta_prob=False)
    inp = _inputs(B=1, T=5, H=1, K=4, V=3, seed=12)
    dfinal = np.zeros((1, 1, 3, 4))
    dfinal[0, 0, 1, 2] = 1.0
    gr = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], np.zeros((1, 5, 1, 3)),
                             scale=0.5, A_log=inp["A_log"], dt_bias=inp["dt_bias"],
                             initial_state=inp["initial_state"], dfinal=dfinal, **mode)
    M = np.eye(4)
    for t in range(5):
        z = inp["g"][0, t, 0].numpy() + inp["dt_bias"][0].numpy()
        a = -np.exp(inp["A_log"][0].item()) * (np.maximum(z, 0) + np.log1p(np.exp(-np.abs(z))))
        kt = inp["k"][0, t, 0].numpy()
        kt = kt / np.sqrt(kt @ kt + 1e-6)
        bt = 1 / (1 + np.exp(-inp["beta"][0, t, 0].item()))
        M = M @ (np.diag(np.exp(a)) @ (np.eye(4) - bt * np.outer(kt, kt)))
    expected = np.zeros((3, 4))
    expected[1] = M[:, 2]  # S_T[1, 2] = sum_j S0[1, j] M[j, 2]
    np.testing.assert_allclose(gr["initial_state"][0, 0], expected, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mode", MODES, ids=[m["gate"] + ("_l2" if m["qk_l2norm"] else "") for m in MODES])
@pytest.mark.parametrize("chunk", [4, 5, 64])
def test_chunk_backward_equals_autograd(mode, chunk):
    """The hand-derived chunked backward (oracle/chunk_backward.py) gives the
    autograd gradients of the token recurrence, for every input: chunk sizes
    that cut the sequences into several full and partial chunks, and one
    larger than every sequence; dense with states and a final-state gradient,
    and packed with an empty sequence."""
    gen = torch.Generator().manual_seed(7)
    for kw in (dict(B=2, T=13, H=2, K=6, V=5, seed=11), dict(lengths=[7, 0, 1, 12], H=2, K=6, V=5, seed=12)):
        inp = _prep(_inputs(**kw), mode)
        B, T = inp["q"].shape[:2]
        dout = torch.randn((B, T, 2, 5), generator=gen, dtype=torch.float64).numpy()
        dfin = torch.randn((inp["N"], 2, 5, 6), generator=gen, dtype=torch.float64).numpy()
        args = dict(scale=0.4, A_log=inp["A_log"], dt_bias=inp["dt_bias"], lower_bound=mode["lower_bound"],
                    gate=mode["gate"], beta_prob=mode["beta_prob"], qk_l2norm=mode["qk_l2norm"],
                    initial_state=inp["initial_state"], dfinal=dfin, cu_seqlens=inp["cu_seqlens"])
        ref = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, **args)
        got = oracle.chunk_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, chunk=chunk, **args)
        for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
            if ref[name] is None:
                assert got[name] is None, name
                continue
            scale_ = max(np.abs(ref[name]).max(), 1e-300)
            assert np.abs(got[name] - ref[name]).max() <= 1e-10 * scale_, (name, chunk)


def test_chunk_backward_intermediates():
    """The kept per-chunk dS_end values chain as the reverse recurrence
    dS_prev = scale dO^T Qg + dS Diag(gC) - dU^T W implies: the first chunk's
    incoming dS is the next chunk's ... down to dfinal for the last chunk."""
    inp = _inputs(B=1, T=11, H=1, K=4, V=3, seed=21)
    dout = np.ones((1, 11, 1, 3))
    dfin = np.full((1, 1, 3, 4), 0.25)
    got = oracle.chunk_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, scale=1.0,
                                A_log=inp["A_log"], dt_bias=inp["dt_bias"], initial_state=inp["initial_state"],
                                dfinal=dfin, chunk=4, keep=True)
    chunks = got["chunks"][(0, 0)]
    assert len(chunks) == 3 and chunks[0]["dP"].shape == (4, 4) and chunks[-1]["dP"].shape == (3, 3)
    np.testing.assert_array_equal(chunks[-1]["dS_end"], dfin[0, 0])
