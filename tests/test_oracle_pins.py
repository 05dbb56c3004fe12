"""Pins of the fp64 CPU oracle against facts fixed outside the oracle itself.

The pages ("Interdomain Attention: Beyond Token-Level Key-Value Memory") print
no worked numeric example, so the oracle is pinned by closed forms, reductions
to textbook/library routines, invariants and brute force on tiny inputs.  Each
test names the plausible oracle mistake it would catch.
"""
import math
from pathlib import Path

import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import ida_oracle as orc
from linear_token_mixer_sc_gb300 import inputs

GOLDEN = Path(__file__).parent / "golden"


def _rand_unit(rng, N, R, d, W):
    q = rng.standard_normal((N, R))
    k = rng.standard_normal((N, R))
    v = rng.standard_normal((N, d))
    wq = rng.standard_normal((R, W)) * 0.5
    wk = rng.standard_normal((R, W)) * 0.5
    nw = 1.0 + 0.3 * rng.standard_normal(R + d)
    bs = 0.3 * rng.standard_normal(R + d)
    return q, k, v, wq, wk, nw, bs


def _rand_modes(rng, M, complex_b=True):
    r = rng.uniform(0.5, 0.99, M)
    th = rng.uniform(-math.pi, math.pi, M)
    lam = r * np.exp(1j * th)
    if complex_b:
        Bv = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    else:
        Bv = np.ones(M, dtype=complex)
    return lam, Bv


# ---- a1: causal depthwise conv ------------------------------------------

def test_conv_is_numpy_causal_convolution():
    """Tap order / causality / padding: equals np.convolve with reversed taps.

    Catches reversed taps (cross-correlation vs convolution), a look-ahead
    (non-causal) index, and wrong zero padding.
    """
    rng = np.random.default_rng(0)
    N, C, W = 37, 5, 4
    x = rng.standard_normal((N, C))
    w = rng.standard_normal((C, W))
    s = orc.causal_conv(x, w)
    for c in range(C):
        ref = np.convolve(x[:, c], w[c, ::-1])[:N]
        np.testing.assert_allclose(s[:, c], ref, rtol=1e-13, atol=1e-13)


def test_conv_tail_is_history():
    """A carried tail acts as the W-1 rows before position 0."""
    rng = np.random.default_rng(1)
    N, C, W = 9, 3, 4
    x = rng.standard_normal((N + W - 1, C))
    w = rng.standard_normal((C, W))
    full = orc.causal_conv(x, w)
    part = orc.causal_conv(x[W - 1:], w, tail=x[:W - 1])
    np.testing.assert_allclose(part, full[W - 1:], rtol=1e-13, atol=1e-13)


# ---- a2: SiLU and the feature map ---------------------------------------

def test_silu_matches_logistic():
    """SiLU(x) = x * sigmoid(x) (scipy's expit), and sigma(ln 3) = 3/4."""
    for x in (-30.0, -3.0, -0.5, 0.0, 1e-8, 0.7, 4.0, 50.0):
        assert orc.silu(x) == pytest.approx(x * expit(x), rel=1e-14, abs=1e-300)
    assert orc.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)


def test_feature_map_squared_norm_invariants():
    """xi = f / (|f|^2 + eps), f = SiLU(s): parallel to f, <xi, f> ~ 1.

    With an l2 (unsquared) norm <xi, f> would be |f| instead of ~1; with no
    normalisation it would be |f|^2.
    """
    rng = np.random.default_rng(2)
    s = rng.standard_normal((20, 16)) * 2.0
    xi = orc.feature_map(s)
    f = s * expit(s)
    n2 = (f * f).sum(1)
    np.testing.assert_allclose((xi * f).sum(1), n2 / (n2 + 1e-6), rtol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(xi, axis=1), np.sqrt(n2) / (n2 + 1e-6), rtol=1e-13)
    cos = (xi * f).sum(1) / (np.linalg.norm(xi, axis=1) * np.sqrt(n2))
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)


def test_feature_map_l2_invariants():
    """The l_2 reading, xi = f / (|f| + eps): parallel to f with |xi| = |f| / (|f| + eps).

    With the squared norm |xi| would be ~1/|f|; without the epsilon or with it under
    a square root the norm identity breaks at small |f|."""
    rng = np.random.default_rng(21)
    s = rng.standard_normal((20, 16)) * 2.0
    s[3] *= 1e-4  # a row with tiny |f|, where the epsilon placement shows
    xi = orc.feature_map(s, l2=True)
    f = s * expit(s)
    n = np.sqrt((f * f).sum(1))
    np.testing.assert_allclose(np.linalg.norm(xi, axis=1), n / (n + 1e-6), rtol=1e-12)
    cos = (xi * f).sum(1) / (np.linalg.norm(xi, axis=1) * n)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)


def test_feature_map_l2_flag_reaches_both_feature_maps():
    """With FEAT_L2 the forward uses the l_2 map for q (the readout scales with it) and for
    k (only through the RMSNorm epsilon); lambda = 1, B = 1, M = 1 reduces the readout to
    cumulative sums of those features."""
    rng = np.random.default_rng(22)
    N, R, d, W = 25, 4, 3, 3
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    one = np.array([1.0 + 0j])
    out, _, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, one, one, flags=orc.FEAT_L2)
    xq = orc.feature_map(orc.causal_conv(q, wq), l2=True)
    kt = orc.rmsnorm_affine(orc.feature_map(orc.causal_conv(k, wk), l2=True), nw[:R], bs[:R])
    vt = orc.rmsnorm_affine(v, nw[R:], bs[R:])
    ref = (xq * np.cumsum(kt, 0)).sum(1)[:, None] * np.cumsum(vt, 0)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-11)
    plain, _, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, one, one)
    assert np.abs(plain - out).max() > 1e-3 * np.abs(out).max()


def test_rmsnorm_unit_mean_square_and_affine():
    """mean(y^2) = ms/(ms+eps) with w=1,b=0; affine applied after the norm."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 12)) * 3.0
    y = orc.rmsnorm_affine(x, np.ones(12), np.zeros(12))
    ms = (x * x).mean(1)
    np.testing.assert_allclose((y * y).mean(1), ms / (ms + 1e-6), rtol=1e-13)
    w = rng.standard_normal(12)
    b = rng.standard_normal(12)
    y2 = orc.rmsnorm_affine(x, w, b)
    np.testing.assert_allclose(y2, y * w + b, rtol=1e-13, atol=1e-14)


def test_rmsnorm_hand_value():
    """x = (3, 4): mean square 12.5, so y = x / sqrt(12.5 + 1e-6)."""
    y = orc.rmsnorm_affine(np.array([[3.0, 4.0]]), np.array([1.0, 1.0]), np.array([0.0, 0.0]))
    np.testing.assert_allclose(y[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-6), rtol=1e-15)


def test_prologue_golden_worked_example():
    """Hand-derived values (tests/golden/prologue_R2_W2.txt) of conv, xi, RMSNorm."""
    L = math.log(3.0)
    g = (L / 2) * math.sqrt(3.0) / (math.sqrt(3.0) + 1.0)
    env = {"L": L, "g": g, "n0": 0.625 * L * L + 1e-6, "n1": g * g + L * L / 16 + 1e-6,
           "sqrt": math.sqrt}
    exp = {}
    for line in (GOLDEN / "prologue_R2_W2.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        name, t, c, expr = line.split(None, 3)
        exp[(name, int(t), int(c))] = eval(expr, {"__builtins__": {}}, env)
    w = np.array([[0.5, 1.0], [1.0, -1.0]])
    x = np.array([[L, L], [0.0, 2 * L]])
    s = orc.causal_conv(x, w)
    xi = orc.feature_map(s)
    y = orc.rmsnorm_affine(xi, np.array([2.0, 0.5]), np.array([0.1, -0.2]))
    got = {"s": s, "xi": xi, "y": y}
    assert len(exp) == 12
    for (name, t, c), val in exp.items():
        assert got[name][t, c] == pytest.approx(val, rel=1e-12, abs=1e-14), (name, t, c)


def test_unit_feature_wiring():
    """q: conv+xi, no RMSNorm; k: conv+xi+RMSNorm(key half); v: RMSNorm(value half), no conv."""
    rng = np.random.default_rng(4)
    N, R, d, W = 11, 6, 5, 4
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    xq, kt, vt = orc.unit_features(q, k, v, wq, wk, nw, bs)
    np.testing.assert_allclose(xq, orc.feature_map(orc.causal_conv(q, wq)), rtol=1e-14)
    np.testing.assert_allclose(
        kt, orc.rmsnorm_affine(orc.feature_map(orc.causal_conv(k, wk)), nw[:R], bs[:R]), rtol=1e-14)
    np.testing.assert_allclose(vt, orc.rmsnorm_affine(v, nw[R:], bs[R:]), rtol=1e-14)


# ---- a4-a7: recurrence and readout --------------------------------------

def _double_sum(xq, kt, vt, lam, Bv):
    """o_t = Re sum_m sum_{s,s'<=t} lam^{t-s} lam^{t-s'} B^2 (xq_t.kt_s) vt_{s'}."""
    N = xq.shape[0]
    out = np.zeros((N, vt.shape[1]))
    den = np.zeros(N)
    for t in range(N):
        s = np.arange(t + 1)
        P = lam[None, :] ** (t - s)[:, None]            # [s, m]
        g = kt[: t + 1] @ xq[t]                          # [s]
        a = Bv * (P * g[:, None]).sum(0)                 # [m]
        Gam = Bv[:, None] * (P.T @ vt[: t + 1])          # [m, d]
        eta = Bv * P.sum(0)                              # [m]
        out[t] = (a[:, None] * Gam).sum(0).real
        den[t] = (a * eta).sum().real
    return out, den


def test_recurrence_equals_bruteforce_double_sum():
    """Step recurrence == closed-form double sum (complex lambda and B).

    Catches a conjugated lambda or B, B instead of B^2, a factor 2, taking the
    real part early, or an off-by-one in the decay powers.
    """
    rng = np.random.default_rng(5)
    N, R, d, M, W = 24, 5, 3, 4, 4
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    lam, Bv = _rand_modes(rng, M)
    out, den, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, lam, Bv)
    xq, kt, vt = orc.unit_features(q, k, v, wq, wk, nw, bs)
    ref, rden = _double_sum(xq, kt, vt, lam, Bv)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(den, rden, rtol=1e-10, atol=1e-12)
    out_e, _, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, lam, Bv, flags=orc.READOUT_ETA)
    np.testing.assert_allclose(out_e, ref / rden[:, None], rtol=1e-9, atol=1e-12)


def test_lambda_one_single_mode_is_cumulative_sums():
    """lambda = 1, B = 1, M = 1: o_t = (xq_t . cumsum kt) * cumsum vt."""
    rng = np.random.default_rng(6)
    N, R, d, W = 30, 4, 3, 2
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    out, _, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, np.array([1.0 + 0j]), np.array([1.0 + 0j]))
    xq, kt, vt = orc.unit_features(q, k, v, wq, wk, nw, bs)
    ref = (xq * np.cumsum(kt, 0)).sum(1)[:, None] * np.cumsum(vt, 0)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-11)


def test_lambda_zero_is_memoryless():
    """lambda = 0: o_t = Re(sum_m B_m^2) (xq_t . kt_t) vt_t."""
    rng = np.random.default_rng(7)
    N, R, d, M, W = 13, 4, 5, 3, 3
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    Bv = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    out, _, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, np.zeros(M, complex), Bv)
    xq, kt, vt = orc.unit_features(q, k, v, wq, wk, nw, bs)
    ref = (Bv ** 2).sum().real * (xq * kt).sum(1)[:, None] * vt
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("C", [1, 7, 16, 64, 50])
def test_chunked_form_matches_recurrence(C):
    """Chunk re-association: same outputs and final state for any chunk length."""
    rng = np.random.default_rng(8)
    N, R, d, M, W = 50, 6, 4, 5, 4
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    lam, Bv = _rand_modes(rng, M)
    out, den, st = orc.unit_forward(q, k, v, wq, wk, nw, bs, lam, Bv)
    xq, kt, vt = orc.unit_features(q, k, v, wq, wk, nw, bs)
    out_c, den_c, st_c = orc.unit_forward_chunked(xq, kt, vt, lam, Bv, C)
    np.testing.assert_allclose(out_c, out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(den_c, den, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(st_c, st, rtol=1e-11, atol=1e-12)


def test_chunked_from_nonzero_state():
    rng = np.random.default_rng(9)
    N, R, d, M = 21, 3, 3, 4
    xq, kt, vt = rng.standard_normal((N, R)), rng.standard_normal((N, R)), rng.standard_normal((N, d))
    lam, Bv = _rand_modes(rng, M)
    st0 = rng.standard_normal(2 * M * (R + d) + 2 * M)
    a = orc.unit_forward_chunked(xq, kt, vt, lam, Bv, 1, state=st0)
    b = orc.unit_forward_chunked(xq, kt, vt, lam, Bv, 8, state=st0)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-12)


def test_eta_readout_returns_constant_values():
    """eta variant with the same v row at every position returns vt exactly."""
    rng = np.random.default_rng(10)
    N, R, d, M, W = 40, 6, 5, 7, 4
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    v[:] = v[0]
    lam, Bv = _rand_modes(rng, M)
    out, den, _ = orc.unit_forward(q, k, v, wq, wk, nw, bs, lam, Bv, flags=orc.READOUT_ETA)
    vt0 = orc.rmsnorm_affine(v[:1], nw[R:], bs[R:])[0]
    assert np.min(np.abs(den)) > 1e-6
    np.testing.assert_allclose(out, np.broadcast_to(vt0, out.shape), rtol=1e-8, atol=1e-10)


def test_state_is_fixed_size_and_decays():
    """|lambda| < 1: the effect of an early token on the state decays as |lambda|^t."""
    rng = np.random.default_rng(11)
    N, R, d, M, W = 60, 4, 4, 3, 4
    q, k, v, wq, wk, nw, bs = _rand_unit(rng, N, R, d, W)
    lam = np.array([0.5, 0.6 + 0.2j, -0.7])
    Bv = np.ones(M, complex)
    _, _, st1 = orc.unit_forward(q, k, v, wq, wk, nw, bs, lam, Bv)
    v2 = v.copy()
    v2[0] += 1.0
    _, _, st2 = orc.unit_forward(q, k, v2, wq, wk, nw, bs, lam, Bv)
    assert st1.shape == (2 * M * (R + d) + 2 * M,)
    diff = np.abs(st1 - st2).max()
    assert 0 < diff < 0.7 ** (N - 2) * 10


# ---- batched entry points -----------------------------------------------

def _small_problem(dtype="f32", B=2, N=19, H=3, R=8, d=6, M=5, W=4, seed=12):
    p = inputs.make_params(H, R, d, M, W, seed)
    q, k, v = inputs.make_qkv(B, N, H, R, d, dtype, seed)
    return q, k, v, p


def test_batched_forward_matches_unit_forward():
    q, k, v, p = _small_problem()
    res = orc.forward(q, k, v, p, final_state=True)
    B, N, H, R = q.shape
    for b in range(B):
        for h in range(H):
            lam = p["lambda"][h, :, 0] + 1j * p["lambda"][h, :, 1]
            Bv = p["Bvec"][h, :, 0] + 1j * p["Bvec"][h, :, 1]
            out, _, st = orc.unit_forward(q[b, :, h].double().numpy(), k[b, :, h].double().numpy(),
                                          v[b, :, h].double().numpy(), p["conv_w"][0, h],
                                          p["conv_w"][1, h], p["norm_w"][h], p["bias"][h],
                                          lam.astype(np.complex128), Bv.astype(np.complex128))
            np.testing.assert_array_equal(res["out"][b, :, h], out)
            np.testing.assert_array_equal(res["final_state"][b, h, : st.size], st)


def test_units_subset_matches_full():
    q, k, v, p = _small_problem()
    full = orc.forward(q, k, v, p, flags=orc.READOUT_ETA, final_state=True)
    sub = orc.forward(q, k, v, p, flags=orc.READOUT_ETA, final_state=True, units=[4, 1])
    for u in (4, 1):
        b, h = divmod(u, 3)
        np.testing.assert_array_equal(sub["out"][b, :, h], full["out"][b, :, h])
        np.testing.assert_array_equal(sub["final_state"][b, h], full["final_state"][b, h])
    assert np.isnan(sub["out"][0, :, 0]).all()


def test_bf16_bytes_are_read_exactly():
    """bf16 input bytes upcast exactly: same result as their fp32 values."""
    q, k, v, p = _small_problem("bf16")
    a = orc.forward(q, k, v, p)["out"]
    b = orc.forward(q.float(), k.float(), v.float(), p)["out"]
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("j", [1, 3, 7])
def test_prefill_then_decode_equals_longer_prefill(j):
    """prefill(N) == prefill(N-j) + j decode steps: outputs and final state.

    Pins the conv-tail carry (oldest first) and the in-place state layout.
    """
    q, k, v, p = _small_problem(N=17, W=4)
    N = q.shape[1]
    full = orc.forward(q, k, v, p, flags=orc.READOUT_ETA, final_state=True)
    part = orc.forward(q[:, : N - j], k[:, : N - j], v[:, : N - j], p, flags=orc.READOUT_ETA,
                       final_state=True)
    st = part["final_state"].copy()
    for i in range(N - j, N):
        r = orc.decode_step(q[:, i], k[:, i], v[:, i], p, st, flags=orc.READOUT_ETA)
        np.testing.assert_allclose(r["out"], full["out"][:, i], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(st, full["final_state"], rtol=1e-10, atol=1e-12)


def test_short_prefill_tail_is_zero_padded():
    """N < W-1: the tail holds zeros for positions before 0."""
    q, k, v, p = _small_problem(N=2, W=4, R=4, d=4, M=2)
    res = orc.forward(q, k, v, p, final_state=True)
    B, N, H, R = q.shape
    S = res["final_state"].shape[2]
    M, d = 2, 4
    tail_q = res["final_state"][:, :, 2 * M * (R + d) + 2 * M:][:, :, : 3 * R].reshape(B, H, 3, R)
    np.testing.assert_array_equal(tail_q[:, :, 0], 0.0)
    np.testing.assert_array_equal(tail_q[:, :, 1:], q.double().numpy().transpose(0, 2, 1, 3))
    assert S == 2 * M * (R + d) + 2 * M + 2 * 3 * R


# ---- prefill from an initial state ------------------------------------------

@pytest.mark.parametrize("N1,W", [(1, 4), (2, 4), (7, 4), (5, 2), (3, 1)])
def test_prefill_from_state_equals_one_longer_prefill(N1, W):
    """prefill(N1) then prefill(rest, state_in = its final state) == prefill(N):
    the state, eta and raw conv tails carry everything the recurrence and the
    causal conv need, so the outputs after N1 and the final state agree exactly.

    Catches a starting state that is ignored, tails taken at the wrong offset or
    in the wrong order, and final tails that do not reach back into the starting
    tails when the second part is shorter than W-1."""
    for N in (N1 + 1, N1 + 2, N1 + 9):
        q, k, v, p = _small_problem(N=N, W=W)
        full = orc.forward(q, k, v, p, flags=orc.READOUT_ETA, final_state=True)
        a = orc.forward(q[:, :N1], k[:, :N1], v[:, :N1], p, flags=orc.READOUT_ETA, final_state=True)
        b = orc.forward(q[:, N1:], k[:, N1:], v[:, N1:], p, flags=orc.READOUT_ETA, final_state=True,
                        state_in=a["final_state"])
        np.testing.assert_array_equal(b["out"], full["out"][:, N1:])
        np.testing.assert_array_equal(b["final_state"], full["final_state"])


def test_prefill_from_state_one_position_is_decode_step():
    """A one-position prefill from a state equals one decode step from it (the
    decode step is a separate code path: in-place state, tail shift)."""
    q, k, v, p = _small_problem(N=6, W=4)
    st = orc.forward(q[:, :5], k[:, :5], v[:, :5], p, final_state=True)["final_state"]
    r = orc.forward(q[:, 5:], k[:, 5:], v[:, 5:], p, flags=orc.READOUT_ETA, final_state=True, state_in=st)
    st2 = st.copy()
    dec = orc.decode_step(q[:, 5], k[:, 5], v[:, 5], p, st2, flags=orc.READOUT_ETA)
    np.testing.assert_allclose(r["out"][:, 0], dec["out"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["final_state"], st2, rtol=1e-12, atol=1e-14)
