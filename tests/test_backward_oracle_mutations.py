"""The chunked backward oracle's pin is sensitive: plant a plausible mistake
in a copy of ``oracle/chunk_backward.py`` (on the CPU) and check that its
gradients no longer equal the autograd gradients of the token recurrence.

Each mutation is a one-line textual change: a dropped term, a wrong sign, a
missing mask or factor, a transposed operand, a cumulative sum in the wrong
direction.
"""
import importlib.util
import os

import numpy as np
import pytest
import torch

import oracle
from tests.test_backward_oracle import MODES, _inputs, _prep

SRC = os.path.join(os.path.dirname(oracle.__file__), "chunk_backward.py")

MUTATIONS = {
    "dU without the output term": ('dU = scale * c["P"].T @ dO + c["Khat"] @ dS.T', 'dU = c["Khat"] @ dS.T'),
    "state gradient not decayed": ('+ dS * c["gC"][None, :] - dU.T @ c["W"]', '+ dS - dU.T @ c["W"]'),
    "wrong sign of the W term": ('+ dS * c["gC"][None, :] - dU.T @ c["W"]', '+ dS * c["gC"][None, :] + dU.T @ c["W"]'),
    "dP without the output scale": ('dP = np.tril(scale * dO @ c["Unew"].T)', 'dP = np.tril(dO @ c["Unew"].T)'),
    "dT with transposed V product": ('dT = np.tril(dU @ c["Vc"].T + dW @ c["Kg"].T)',
                                     'dT = np.tril(c["Vc"] @ dU.T + dW @ c["Kg"].T)'),
    "dbeta without the T term": ('db = np.einsum("ji,ji->i", Minv, dT)', 'db = 0.0 * np.einsum("ji,ji->i", Minv, dT)'),
    "dM without beta": ('dA = np.tril(-Minv.T @ (dT * b[None, :]) @ Minv.T, -1)', 'dA = np.tril(-Minv.T @ dT @ Minv.T, -1)'),
    "dG without beta": ('dG = dA * b[:, None]', 'dG = dA'),
    "pairwise Gamma sign": ('dGam = tG.sum(1) - tG.sum(0) + tP.sum(1) - tP.sum(0)',
                            'dGam = tG.sum(1) + tG.sum(0) + tP.sum(1) - tP.sum(0)'),
    "Khat scaling term dropped from dGamma": ('- dKhat * c["Khat"]', '- 0.0 * dKhat'),
    "Gamma_C terms dropped": ('dGam[-1] += (dKhat * c["Khat"]).sum(0) + dgC * c["gC"]', 'dGam[-1] += 0.0'),
    "cumulative sum forward": ('da = np.cumsum(dGam[::-1], axis=0)[::-1]', 'da = np.cumsum(dGam, axis=0)'),
    "norm derivative without the projection": (
        'dq[c0:c1, h] = c["rq"] * (dQh - Qh * (Qh * dQh).sum(-1, keepdims=True))', 'dq[c0:c1, h] = c["rq"] * dQh'),
    "sigmoid derivative dropped": ('db if beta_prob else db * b * (1.0 - b)', 'db'),
    "unsafe gate derivative sign": ('return -m * _sigmoid(z), a', 'return m * _sigmoid(z), a'),
    "initial-state gradient not propagated": ('dinit[n, h] = dS', 'dinit[n, h] = 0.0 * dS'),
    "dKg dropped": ('dKh += dKg * eG + dKhat', 'dKh += dKhat'),
    "dV uses T instead of its transpose": ('dv[c0:c1, h] = c["T"].T @ dU', 'dv[c0:c1, h] = c["T"] @ dU'),
}


def _load(src_text, tmp_path, tag):
    path = tmp_path / f"chunk_backward_{tag}.py"
    path.write_text(src_text)
    spec = importlib.util.spec_from_file_location(f"oracle._mutated_{tag}", str(path))
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"  # its relative import of the gate
    spec.loader.exec_module(mod)
    return mod.chunk_backward


def _differs(fn):
    """True if fn's gradients differ from the autograd oracle's on any case."""
    gen = torch.Generator().manual_seed(5)
    for mode in MODES:
        inp = _prep(_inputs(B=2, T=11, H=1, K=5, V=4, seed=31), mode)
        dout = torch.randn((2, 11, 1, 4), generator=gen, dtype=torch.float64).numpy()
        dfin = torch.randn((2, 1, 4, 5), generator=gen, dtype=torch.float64).numpy()
        args = dict(scale=0.6, A_log=inp["A_log"], dt_bias=inp["dt_bias"], lower_bound=mode["lower_bound"],
                    gate=mode["gate"], beta_prob=mode["beta_prob"], qk_l2norm=mode["qk_l2norm"],
                    initial_state=inp["initial_state"], dfinal=dfin)
        ref = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, **args)
        got = fn(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, chunk=4, **args)
        for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
            if ref[name] is None:
                continue
            if np.abs(got[name] - ref[name]).max() > 1e-8 * max(np.abs(ref[name]).max(), 1e-30):
                return True
    return False


def test_unmutated_copy_matches(tmp_path):
    assert not _differs(_load(open(SRC).read(), tmp_path, "clean"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {name}"
    assert _differs(_load(src.replace(old, new), tmp_path, "m")), f"pin missed: {name}"
