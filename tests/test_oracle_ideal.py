"""Pins of the ideal-derivation oracle (oracle/ida_ideal.py): random Fourier features
(Eqs. 5-6), finite-feature kernel regression (Eqs. 3-4) and the interdomain layer of
Fig. 1b on those features, each checked against something other than itself."""
import numpy as np
import pytest

from linear_token_mixer_sc_gb300 import inputs
from oracle import ida_ideal as ii


def test_fourier_features_have_unit_norm():
    """cos^2 + sin^2 = 1 for every frequency, so ||xi(x)||^2 = 1 exactly: K(x, x) = 1."""
    rng = np.random.default_rng(1)
    om = rng.standard_normal((37, 5))
    f = ii.rff(rng.standard_normal((9, 5)) * 3, om)
    np.testing.assert_allclose((f * f).sum(-1), 1.0, rtol=1e-14)


def test_fourier_features_are_shift_invariant_and_match_the_kernel():
    """Bochner (Eq. 5): xi(x).xi(y) depends on x - y only, and averages to the Gaussian
    kernel exp(-||x - y||^2 / 2) for omega ~ N(0, I); with D = 40000 frequencies the
    Monte-Carlo error is about D^-1/2."""
    rng = np.random.default_rng(2)
    D, R = 40000, 4
    om = rng.standard_normal((D, R))
    x = rng.standard_normal((6, R)) * 0.7
    y = rng.standard_normal((6, R)) * 0.7
    got = ii.rff(x, om) @ ii.rff(y, om).T
    shift = rng.standard_normal(R)
    np.testing.assert_allclose(ii.rff(x + shift, om) @ ii.rff(y + shift, om).T, got, atol=1e-12)
    np.testing.assert_allclose(got, ii.gaussian_kernel(x, y), atol=5.0 / np.sqrt(D))


def test_gaussian_kernel_closed_form():
    x = np.array([[0.0, 0.0], [1.0, 2.0]])
    y = np.array([[0.0, 1.0]])
    np.testing.assert_allclose(ii.gaussian_kernel(x, y)[:, 0], [np.exp(-0.5), np.exp(-1.0)], rtol=1e-15)


def test_linear_attention_approaches_kernel_regression():
    """Eq. 4 with Fourier features approaches Eq. 1 with the Gaussian kernel as D grows."""
    rng = np.random.default_rng(3)
    N, R, d = 12, 3, 2
    q, k = rng.standard_normal((N, R)) * 0.5, rng.standard_normal((N, R)) * 0.5
    v = rng.standard_normal((N, d))
    exact = ii.kernel_regression(q, k, v)
    errs = []
    for D in (100, 10000):
        om = np.random.default_rng(4).standard_normal((D, R))
        got = ii.linear_attention(ii.rff(q, om), ii.rff(k, om), v)
        errs.append(np.abs(got - exact).max())
    assert errs[1] < 0.05 and errs[1] < errs[0]


def test_linear_attention_equals_its_recurrent_form():
    """Eq. 4 by its definition equals the running sums S_i = sum fk_n v_n^T, z_i = sum fk_n."""
    rng = np.random.default_rng(5)
    N, F, d = 20, 8, 3
    fq, fk = rng.random((N, F)) + 0.1, rng.random((N, F)) + 0.1
    v = rng.standard_normal((N, d))
    S = np.zeros((F, d))
    z = np.zeros(F)
    rec = np.zeros((N, d))
    for i in range(N):
        S += np.outer(fk[i], v[i])
        z += fk[i]
        rec[i] = fq[i] @ S / (fq[i] @ z)
    np.testing.assert_allclose(ii.linear_attention(fq, fk, v), rec, rtol=1e-12)


def _unit(seed, N=9, R=3, D=4, d=2, M=3):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((N, R)), rng.standard_normal((N, R)), rng.standard_normal((N, d))
    om = rng.standard_normal((D, R))
    lam = 0.9 * np.exp(1j * rng.uniform(-1, 1, M))
    B = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    return q, k, v, om, lam, B


def test_ideal_layer_equals_its_closed_form():
    """The recurrence and ratio readout equal the closed-form double sums
    num_t = Re sum_m sum_{s,s'} lam^(t-s) lam^(t-s') B^2 (xi_q . xi_k_s) v_s',
    den_t = Re sum_m sum_{s,s'} lam^(t-s) lam^(t-s') B^2 (xi_q . xi_k_s), brute force."""
    q, k, v, om, lam, B = _unit(6)
    fq, fk = ii.rff(q, om), ii.rff(k, om)
    got = ii.ideal_unit(q, k, v, om, lam, B)
    N = q.shape[0]
    for t in range(N):
        num = np.zeros(v.shape[1])
        den = 0.0
        for m in range(lam.shape[0]):
            for s in range(t + 1):
                for s2 in range(t + 1):
                    w = lam[m] ** (t - s) * lam[m] ** (t - s2) * B[m] ** 2 * (fq[t] @ fk[s])
                    num += (w * v[s2]).real
                    den += w.real
        np.testing.assert_allclose(got[t], num / den, rtol=1e-9, atol=1e-12)


def test_ideal_layer_returns_a_constant_value():
    """The ratio readout of a constant value row returns that row (Eq. 4's normalisation,
    kept by the eta normaliser)."""
    q, k, v, om, lam, B = _unit(7)
    v[:] = v[0]
    np.testing.assert_allclose(ii.ideal_unit(q, k, v, om, lam, B), np.broadcast_to(v[0], v.shape), rtol=1e-10)


def test_ideal_layer_with_one_unit_mode_is_the_running_mean():
    """lambda = 1, M = 1, B = 1: o_t = (xi_q . sum xi_k)(sum v) / ((xi_q . sum xi_k)(t + 1))."""
    q, k, v, om, _, _ = _unit(8)
    got = ii.ideal_unit(q, k, v, om, np.ones(1, complex), np.ones(1, complex))
    mean = np.cumsum(v, 0) / np.arange(1, v.shape[0] + 1)[:, None]
    np.testing.assert_allclose(got, mean, rtol=1e-10)


def test_forward_wiring_and_omega_draw():
    """The batched forward maps [B, N, H, *] units with per-head frequencies; the draw
    is seeded and has the stated variance."""
    B, N, H, R, D, d, M = 2, 5, 2, 4, 3, 2, 2
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((B, N, H, c)) for c in (R, R, d))
    om = inputs.make_omega(H, D, R, seed=3)
    assert om.shape == (H, D, R) and om.dtype == np.float32
    np.testing.assert_array_equal(om, inputs.make_omega(H, D, R, seed=3))
    big = inputs.make_omega(1, 4000, 16, seed=1)
    assert abs(big.var() * 16 - 1.0) < 0.05
    lam = np.stack([np.full((H, M), 0.8), np.zeros((H, M))], -1)
    Bv = np.stack([np.ones((H, M)), np.zeros((H, M))], -1)
    out = ii.ideal_forward(q, k, v, om, lam, Bv)
    for b in range(B):
        for h in range(H):
            ref = ii.ideal_unit(q[b, :, h], k[b, :, h], v[b, :, h], om[h], lam[h, :, 0] + 0j, Bv[h, :, 0] + 0j)
            np.testing.assert_allclose(out[b, :, h], ref, rtol=1e-12)


MUTATIONS = [
    ("np.concatenate([np.cos(th), np.sin(th)], axis=-1) / np.sqrt(D)",
     "np.concatenate([np.cos(th), np.cos(th)], axis=-1) / np.sqrt(D)"),      # sine half dropped
    ("np.concatenate([np.cos(th), np.sin(th)], axis=-1) / np.sqrt(D)",
     "np.concatenate([np.cos(th), np.sin(th)], axis=-1) / D"),               # wrong normalisation
    ("U = lam[:, None] * U + B[:, None] * fk[t][None, :]",
     "U = np.conj(lam)[:, None] * U + B[:, None] * fk[t][None, :]"),          # conjugated decay
    ("eta = lam * eta + B", "eta = lam * eta + 1"),                           # eta without B
    ("a = U @ fq[t]", "a = U @ fk[t]"),                                       # key features read out
    ("w = fk[: i + 1] @ fq[i]", "w = fq[: i + 1] @ fq[i]"),                   # Eq. 4 weights from the queries
]


@pytest.mark.parametrize("old,new", MUTATIONS, ids=range(len(MUTATIONS)))
def test_planted_mistakes_are_caught(old, new, monkeypatch):
    """Each planted mistake in a copy of the oracle makes at least one pin above fail."""
    import importlib.util
    import sys
    import types
    src = open(ii.__file__).read()
    assert old in src
    mod = types.ModuleType("ida_ideal_mutant")
    exec(compile(src.replace(old, new, 1), "ida_ideal_mutant", "exec"), mod.__dict__)
    monkeypatch.setattr(sys.modules[__name__], "ii", mod)
    pins = [test_fourier_features_have_unit_norm, test_fourier_features_are_shift_invariant_and_match_the_kernel,
            test_linear_attention_approaches_kernel_regression, test_linear_attention_equals_its_recurrent_form,
            test_ideal_layer_equals_its_closed_form, test_ideal_layer_returns_a_constant_value,
            test_ideal_layer_with_one_unit_mode_is_the_running_mean]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0
