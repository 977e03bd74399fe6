"""Pins for the fp64 oracle: each check ties it to something other than itself.

* a hand-derived worked example (tests/golden/worked_example.json),
* brute force: the explicit O(N^2) masked form against the S/Z recurrence,
* closed forms and invariants the paper's formulas imply (constant V, positive
  normalizers, non-causal = causal at i = N, key-order invariance, causality),
* the degree-2 polynomial kernel, whose exact feature map turns the associative
  path into an explicit kernel sum,
* random Fourier features, whose inner products estimate the RBF kernel
  (a Monte Carlo check at many features),
* central finite differences for the cumulative-sum backward,
* prefill + decode steps = causal forward over the concatenated sequence,
* mutation checks: a plausible mistake planted in a copy of the oracle must
  fail at least one of the pins above.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import linear_attention as la

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _num(s):
    s = s.strip()
    neg = s.startswith("-")
    body = s[1:] if neg else s
    if body.startswith("ln"):
        val = math.log(float(body[2:]))
    else:
        val = float(Fraction(body))
    return -val if neg else val


def _arr(x):
    if isinstance(x, str):
        return _num(x)
    return np.array([_arr(e) for e in x], dtype=np.float64)


def _rand(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# --------------------------------------------------------------------------- phi

def test_phi_closed_form():
    assert la.elu_plus_one(0.0) == 1.0
    assert la.elu_plus_one(2.0) == 3.0
    assert la.elu_plus_one(0.5) == 1.5
    assert la.elu_plus_one(-1.0) == pytest.approx(math.exp(-1.0), rel=1e-15)
    assert la.elu_plus_one(-math.log(2.0)) == pytest.approx(0.5, rel=1e-15)
    # continuous at 0 from both sides, strictly positive everywhere
    assert la.elu_plus_one(1e-12) == pytest.approx(1.0, abs=1e-11)
    assert la.elu_plus_one(-1e-12) == pytest.approx(1.0, abs=1e-11)
    x = np.linspace(-30, 30, 2001)
    assert np.all(la.elu_plus_one(x) > 0)


def test_phi_grad_matches_central_differences():
    x = np.concatenate([np.linspace(-6, -1e-3, 50), np.linspace(1e-3, 6, 50)])
    h = 1e-6
    fd = (la.elu_plus_one(x + h) - la.elu_plus_one(x - h)) / (2 * h)
    np.testing.assert_allclose(la.elu_plus_one_grad(x), fd, rtol=1e-8, atol=1e-10)


# ------------------------------------------------------------ worked example

def test_worked_example_phi(golden):
    np.testing.assert_allclose(la.elu_plus_one(_arr(golden["q"])), _arr(golden["phi_q"]), rtol=1e-15)
    np.testing.assert_allclose(la.elu_plus_one(_arr(golden["k"])), _arr(golden["phi_k"]), rtol=1e-15)


def _check_worked_example(mod, golden):
    q, k, v = _arr(golden["q"]), _arr(golden["k"]), _arr(golden["v"])
    want_c = _arr(golden["causal_out"])
    want_nc = _arr(golden["noncausal_out"])
    np.testing.assert_allclose(mod.masked_attention(q, k, v, causal=True), want_c, rtol=1e-14)
    np.testing.assert_allclose(mod.recurrent_attention(q, k, v)[0], want_c, rtol=1e-14)
    np.testing.assert_allclose(mod.masked_attention(q, k, v, causal=False), want_nc, rtol=1e-14)
    out, S, Z = mod.linearized_attention(q, k, v)
    np.testing.assert_allclose(out, want_nc, rtol=1e-14)
    np.testing.assert_allclose(S, _arr(golden["S_N"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(Z, _arr(golden["Z_N"]), rtol=1e-14)
    _, S2, Z2 = mod.prefill(q, k, v)
    np.testing.assert_allclose(S2, _arr(golden["S_N"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(Z2, _arr(golden["Z_N"]), rtol=1e-14)
    dec = golden["decode"]
    o, S3, Z3 = mod.decode_step(_arr(dec["q"]), _arr(dec["k"]), _arr(dec["v"]), S2, Z2)
    np.testing.assert_allclose(S3, _arr(dec["S_new"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(Z3, _arr(dec["Z_new"]), rtol=1e-14)
    np.testing.assert_allclose(o, _arr(dec["out"]), rtol=1e-14)


def test_worked_example(golden):
    _check_worked_example(la, golden)


# ------------------------------------------------------- brute force / forms

@pytest.mark.parametrize("N,D,M", [(1, 4, 4), (17, 5, 7), (64, 32, 32)])
def test_masked_equals_recurrence(N, D, M):
    q, k, v = _rand(1, 2, 3, N, D), _rand(2, 2, 3, N, D), _rand(3, 2, 3, N, M)
    a = la.masked_attention(q, k, v, causal=True)
    b, S, Z = la.recurrent_attention(q, k, v)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.forward(q, k, v, causal=True), a, rtol=1e-12, atol=1e-12)


def test_masked_rows_equal_full_masked_form():
    # every row of a sequence that spans the row-by-row loop's edge cases
    # (first row, last row): an off-by-one in the mask fails here
    N, D, M = 37, 6, 5
    q, k, v = _rand(7, N, D), _rand(8, N, D), _rand(9, N, M)
    full = la.masked_attention(q, k, v, causal=True)
    rows = list(range(N))
    np.testing.assert_allclose(la.masked_attention_rows(q, k, v, rows), full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(la.masked_attention_rows(q, k, v, [N - 1, 0, 5]), full[[N - 1, 0, 5]],
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("N,D,M", [(1, 3, 2), (33, 8, 5)])
def test_masked_equals_linearized_noncausal(N, D, M):
    q, k, v = _rand(4, 2, N, D), _rand(5, 2, N, D), _rand(6, 2, N, M)
    a = la.masked_attention(q, k, v, causal=False)
    b = la.linearized_attention(q, k, v)[0]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.forward(q, k, v, causal=False), a, rtol=1e-12, atol=1e-12)


def test_recurrence_final_state_is_full_sum():
    q, k, v = _rand(7, 3, 20, 6), _rand(8, 3, 20, 6), _rand(9, 3, 20, 5)
    _, S, Z = la.recurrent_attention(q, k, v)
    _, S2, Z2 = la.linearized_attention(q, k, v)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Z, Z2, rtol=1e-12)


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [True, False])
def test_constant_v_gives_constant_output(causal):
    q, k = _rand(10, 2, 40, 8, scale=2.0), _rand(11, 2, 40, 8, scale=2.0)
    c = np.array([0.3, -1.7, 2.5])
    v = np.broadcast_to(c, (2, 40, 3))
    np.testing.assert_allclose(oracle.forward(q, k, v, causal), np.broadcast_to(c, (2, 40, 3)),
                               rtol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_denominators_positive(causal):
    q, k = _rand(12, 4, 100, 16, scale=3.0), _rand(13, 4, 100, 16, scale=3.0)
    den = la.denominators(q, k, causal)
    assert np.all(den > 0)


def test_denominators_match_explicit_sum():
    q, k = _rand(14, 2, 9, 4), _rand(15, 2, 9, 4)
    fq, fk = la.elu_plus_one(q), la.elu_plus_one(k)
    W = np.einsum("bid,bjd->bij", fq, fk)
    np.testing.assert_allclose(la.denominators(q, k, True), np.tril(W).sum(-1), rtol=1e-13)
    np.testing.assert_allclose(la.denominators(q, k, False), W.sum(-1), rtol=1e-13)


def test_noncausal_equals_causal_last_row():
    q, k, v = _rand(16, 3, 25, 7), _rand(17, 3, 25, 7), _rand(18, 3, 25, 4)
    c = oracle.forward(q, k, v, causal=True)
    nc = oracle.forward(q, k, v, causal=False)
    np.testing.assert_allclose(c[:, -1], nc[:, -1], rtol=1e-12)
    assert not np.allclose(c[:, 0], nc[:, 0])


def test_noncausal_key_order_invariance():
    q, k, v = _rand(19, 30, 6), _rand(20, 30, 6), _rand(21, 30, 3)
    perm = np.random.default_rng(22).permutation(30)
    np.testing.assert_allclose(oracle.forward(q, k, v, False),
                               oracle.forward(q, k[perm], v[perm], False), rtol=1e-12)


def test_causality():
    q, k, v = _rand(23, 2, 30, 5), _rand(24, 2, 30, 5), _rand(25, 2, 30, 6)
    base = oracle.forward(q, k, v, True)
    i = 12
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, i + 1:] += 1.0
    k2[:, i + 1:] -= 2.0
    v2[:, i + 1:] *= 3.0
    pert = oracle.forward(q2, k2, v2, True)
    np.testing.assert_array_equal(pert[:, : i + 1], base[:, : i + 1])
    assert not np.allclose(pert[:, i + 1:], base[:, i + 1:])


# ------------------------------------------- degree-2 polynomial special case

def _explicit_poly_attention(q, k, v, causal):
    W = np.einsum("...id,...jd->...ij", q, k) ** 2
    if causal:
        W = np.tril(W)
    return np.einsum("...ij,...jm->...im", W, v) / W.sum(-1)[..., None]


@pytest.mark.parametrize("causal", [True, False])
def test_polynomial_kernel_special_case(causal):
    q, k, v = _rand(26, 2, 24, 5), _rand(27, 2, 24, 5), _rand(28, 2, 24, 3)
    want = _explicit_poly_attention(q, k, v, causal)
    np.testing.assert_allclose(la.masked_attention(q, k, v, causal, feature=la.poly2_feature),
                               want, rtol=1e-11)
    if causal:
        got = la.recurrent_attention(q, k, v, feature=la.poly2_feature)[0]
    else:
        got = la.linearized_attention(q, k, v, feature=la.poly2_feature)[0]
    np.testing.assert_allclose(got, want, rtol=1e-10)


# ------------------------------------------------------- backward: finite diff

def _loss(q, k, v, G, causal):
    return float((oracle.forward(q, k, v, causal) * G).sum())


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def _away_from_zero(a, gap=1e-2):
    return np.where(np.abs(a) < gap, np.sign(a + 1e-30) * gap, a)


def _check_backward_fd(mod_backward, causal, N=7, D=3, M=4, seed=30):
    q = _away_from_zero(_rand(seed, 2, N, D))
    k = _away_from_zero(_rand(seed + 1, 2, N, D))
    v = _rand(seed + 2, 2, N, M)
    G = _rand(seed + 3, 2, N, M)
    dq, dk, dv = mod_backward(q, k, v, G, causal=causal)
    fq = _fd_grad(lambda x: _loss(x, k, v, G, causal), q)
    fk = _fd_grad(lambda x: _loss(q, x, v, G, causal), k)
    fv = _fd_grad(lambda x: _loss(q, k, x, G, causal), v)
    for got, want in ((dq, fq), (dk, fk), (dv, fv)):
        err = np.max(np.abs(got - want)) / np.max(np.abs(want))
        assert err < 1e-6, err


@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_finite_differences(causal):
    _check_backward_fd(la.backward, causal)


def test_backward_fd_wider():
    _check_backward_fd(la.backward, True, N=16, D=4, M=4, seed=40)


def test_backward_shapes_and_first_token():
    # at i = 0 the causal output is v_0 exactly, so dv_0 receives dout_0 plus
    # the later positions' share; q_0 has no influence on any output but out_0
    q, k, v = _rand(50, 5, 4), _rand(51, 5, 4), _rand(52, 5, 3)
    G = np.zeros((5, 3))
    G[0] = [1.0, -2.0, 0.5]
    dq, dk, dv = la.backward(q, k, v, G, causal=True)
    np.testing.assert_allclose(dv[0], G[0], rtol=1e-13)
    np.testing.assert_allclose(dv[1:], 0.0, atol=1e-15)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)


# --------------------------------------------------------------- decode pins

def test_prefill_then_decode_equals_causal_forward():
    B, H, P, T, D, M = 2, 3, 11, 6, 5, 4
    q, k, v = _rand(60, B, H, P + T, D), _rand(61, B, H, P + T, D), _rand(62, B, H, P + T, M)
    full = oracle.forward(q, k, v, True)
    out_p, S, Z = oracle.prefill(q[:, :, :P], k[:, :, :P], v[:, :, :P])
    np.testing.assert_allclose(out_p, full[:, :, :P], rtol=1e-12)
    for t in range(P, P + T):
        o, S, Z = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], S, Z)
        np.testing.assert_allclose(o, full[:, :, t], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ mutation checks

class _Mutant:
    """A copy of the oracle with one planted mistake (CPU only)."""

    def __init__(self, **over):
        self.__dict__.update({n: getattr(la, n) for n in (
            "masked_attention", "recurrent_attention", "linearized_attention",
            "prefill", "decode_step", "backward")})
        self.__dict__.update(over)


def _exclusive_masked(q, k, v, causal=True, feature=la.elu_plus_one):
    fq, fk = feature(q), feature(k)
    W = fq @ np.swapaxes(fk, -1, -2)
    if causal:
        W = np.tril(W, -1) + np.eye(W.shape[-1]) * 1e-300
    return (W @ v) / W.sum(-1, keepdims=True)


def _read_before_update(q, k, v, S, Z):
    fq, fk = la.elu_plus_one(q), la.elu_plus_one(k)
    out = (fq @ S) / (fq @ Z)
    return out, S + np.outer(fk, v), Z + fk


def _no_plus_one_recurrence(q, k, v, S0=None, Z0=None, feature=None):
    return la.recurrent_attention(q, k, v, S0, Z0, feature=lambda x: np.where(x > 0, x, np.exp(x)))


def _transposed_linearized(q, k, v, feature=la.elu_plus_one):
    out, S, Z = la.linearized_attention(q, k, v, feature)
    if S.shape[-1] == S.shape[-2]:
        S = np.swapaxes(S, -1, -2)
        out = (feature(q) @ S) / (feature(q) @ Z[..., None])
    return out, S, Z


@pytest.mark.parametrize("mutant", [
    _Mutant(masked_attention=_exclusive_masked),
    _Mutant(decode_step=_read_before_update),
    _Mutant(recurrent_attention=_no_plus_one_recurrence),
    _Mutant(linearized_attention=_transposed_linearized),
], ids=["exclusive-mask", "decode-read-before-update", "phi-without-plus-one",
        "transposed-state"])
def test_mutants_fail_worked_example(mutant, golden):
    with pytest.raises(AssertionError):
        _check_worked_example(mutant, golden)


def _explicit_backward(q, k, v, G, causal, drop_den=False, wrong_dir=False, drop_phi_grad=False):
    """O(N^2) gradient by explicit sums over (i, j) pairs, with optional planted mistakes."""
    fq, fk = la.elu_plus_one(q), la.elu_plus_one(k)
    N = q.shape[-2]
    W = fq @ np.swapaxes(fk, -1, -2)                    # W[i, j] = phi(q_i) . phi(k_j)
    mask = np.tril(np.ones((N, N))) if causal else np.ones((N, N))
    Wm = W * mask
    den = Wm.sum(-1)                                    # [.., N]
    out = (Wm @ v) / den[..., None]
    gN = G / den[..., None]
    gd = np.zeros(den.shape) if drop_den else -(G * out).sum(-1) / den
    # coefficient of phi(k_j) in d/dphi(q_i) and of phi(q_i) in d/dphi(k_j)
    coef = (gN @ np.swapaxes(v, -1, -2) + gd[..., :, None]) * mask    # [i, j]
    kmask = mask.T if wrong_dir else mask
    coef_k = (gN @ np.swapaxes(v, -1, -2) + gd[..., :, None]) * kmask
    dphiq = coef @ fk
    dphik = np.swapaxes(coef_k, -1, -2) @ fq
    dv = np.swapaxes(Wm if not wrong_dir else W * kmask, -1, -2) @ gN
    if drop_phi_grad:
        return dphiq, dphik, dv
    return dphiq * la.elu_plus_one_grad(q), dphik * la.elu_plus_one_grad(k), dv


@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_explicit_pair_sums(causal):
    q, k, v, G = _rand(70, 2, 13, 4), _rand(71, 2, 13, 4), _rand(72, 2, 13, 5), _rand(73, 2, 13, 5)
    for got, want in zip(la.backward(q, k, v, G, causal), _explicit_backward(q, k, v, G, causal)):
        np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("flaw", ["drop_den", "wrong_dir", "drop_phi_grad"])
def test_mutant_backward_fails_finite_differences(flaw):
    bad = lambda q, k, v, G, causal=True: _explicit_backward(q, k, v, G, causal, **{flaw: True})
    # the unflawed explicit form passes the same check
    _check_backward_fd(lambda q, k, v, G, causal=True: _explicit_backward(q, k, v, G, causal), True)
    with pytest.raises(AssertionError):
        _check_backward_fd(bad, True)


# ------------------------------------------------------- random Fourier features

def test_random_fourier_features_estimate_the_rbf_kernel():
    """E[phi(x) . phi(y)] = exp(-|x - y|^2 / (2 sigma^2)) for W ~ N(0, sigma^-2 I), b ~ U[0, 2 pi):
    with F = 2^17 features the estimate is within a few 1/sqrt(F) of the kernel (checked
    for D != F, so a transposed W cannot pass, and at several distances)."""
    rng = np.random.default_rng(7)
    D, F, sigma = 8, 1 << 17, 1.5
    W = rng.standard_normal((F, D)) / sigma
    b = rng.uniform(0.0, 2.0 * np.pi, F)
    x = rng.standard_normal((6, D)) * 0.6
    y = x + rng.standard_normal((6, D)) * np.array([0.0, 0.2, 0.5, 1.0, 1.5, 2.5])[:, None]
    got = np.sum(la.random_fourier_feature(x, W, b) * la.random_fourier_feature(y, W, b), axis=-1)
    want = np.exp(-np.sum((x - y) ** 2, axis=-1) / (2 * sigma ** 2))
    assert np.max(np.abs(got - want)) < 6.0 / np.sqrt(F)
    assert abs(got[0] - 1.0) < 6.0 / np.sqrt(F)            # x = y: the kernel is 1
    # without the random phases the estimate is a different kernel
    bad = np.sum(np.sqrt(2.0 / F) * np.cos(x @ W.T) * np.sqrt(2.0 / F) * np.cos(y @ W.T), axis=-1)
    assert np.max(np.abs(bad - want)) > 0.05


def test_random_fourier_features_shape_and_scale():
    rng = np.random.default_rng(8)
    W = rng.standard_normal((12, 5))
    b = rng.uniform(0.0, 2.0 * np.pi, 12)
    f = la.random_fourier_feature(rng.standard_normal((3, 4, 5)), W, b)
    assert f.shape == (3, 4, 12)
    assert np.max(np.abs(f)) <= np.sqrt(2.0 / 12) + 1e-15     # each feature is sqrt(2/F) cos(.)
