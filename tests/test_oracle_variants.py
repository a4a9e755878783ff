"""Pins for the variant oracle (oracle/la_variants.c), against things other than itself.

Sources: "Transformers are RNNs" (TaR, read in its Chinese translation) and
"Linear Transformers Are Secretly Fast Weight Programmers" (FWP, read in a
Chinese news summary whose equations were lost; the readings are listed in
the design notes).

  * hand-derived features and sequences in tests/golden/variant_examples.json;
  * the C feature loops vs the vectorised numpy maps (two programs);
  * closed forms: phi(x).phi(y) = (x.y)^2 for the polynomial map (TaR sec.
    3.2.1), the DPFP-1 quadrant property at D = 2 (FWP's figure), unit sums
    under sum normalisation;
  * the sum-update recurrence vs the quadratic definition form, for every
    feature map and read-out;
  * the delta-rule recurrence vs an independent chunked evaluation (the UT
    transform: within a chunk the pseudo-values U solve a unit lower
    triangular system, derived below), at several chunk lengths;
  * delta-rule closed forms: beta = 0 keeps the state, beta = 1 on a one-hot
    key overwrites its slot; split-and-carry equals the whole;
  * every planted mistake breaks at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import definition_variant, features_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "variant_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _ev(e):
    return float(eval(e, {"math": math}))


def _rand(B, N, D, M, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, N, D)) * scale).astype(np.float32)
    k = (rng.standard_normal((B, N, D)) * scale).astype(np.float32)
    v = rng.standard_normal((B, N, M)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=(B, N)).astype(np.float32)
    return q, k, v, beta


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ------------------------------------------------------------------ features

@pytest.mark.parametrize("case", _golden()["features"], ids=lambda c: c["name"])
def test_golden_features(case):
    x = np.array([case["x"]], np.float32)
    want = np.array([_ev(e) for e in case["phi"]])
    got = oracle.features(x, case["fm"], case["nu"], case.get("sumnorm", False))[0]
    assert np.allclose(got, want, rtol=0, atol=1e-15), (got, want)


@pytest.mark.parametrize("fm,nu,D", [("elu1", 1, 16), ("dpfp", 1, 16), ("dpfp", 3, 8), ("dpfp", 2, 64), ("poly2", 1, 16)])
@pytest.mark.parametrize("sumnorm", [False, True])
def test_features_two_programs(fm, nu, D, sumnorm):
    if fm == "poly2" and sumnorm:
        pytest.skip("sum normalisation is defined for non-negative feature maps")
    x = np.random.default_rng(3).standard_normal((40, D)).astype(np.float32)
    a = oracle.features(x, fm, nu, sumnorm)
    b = features_np(x, fm, nu, sumnorm)
    assert a.shape == (40, oracle.feature_dim(fm, D, nu))
    assert np.abs(a - b).max() <= 1e-13 * max(1.0, np.abs(b).max())


def test_poly2_kernel_closed_form():
    """TaR sec. 3.2.1: the degree-2 polynomial kernel (x.y)^2 has an exact feature map."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((30, 16)).astype(np.float32)
    y = rng.standard_normal((30, 16)).astype(np.float32)
    fx, fy = oracle.features(x, "poly2"), oracle.features(y, "poly2")
    want = (x.astype(np.float64) * y.astype(np.float64)).sum(-1) ** 2
    assert np.allclose((fx * fy).sum(-1), want, rtol=1e-12, atol=1e-12)


def test_dpfp_quadrants_d2():
    """FWP's figure: at D = 2, nu = 1 each point has one non-zero feature and the
    four quadrants use four different ones (orthogonal in feature space)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((400, 2)).astype(np.float32)
    f = oracle.features(x, "dpfp", 1)
    nz = (f != 0).sum(-1)
    assert (nz == 1).all()
    idx = f.argmax(-1)
    quad = np.where(x[:, 0] > 0, np.where(x[:, 1] > 0, 0, 3), np.where(x[:, 1] > 0, 1, 2))
    assert (idx == quad).all()
    assert np.allclose(f.max(-1), np.abs(x[:, 0] * x[:, 1]).astype(np.float64))


@pytest.mark.parametrize("fm,nu", [("elu1", 1), ("dpfp", 1), ("dpfp", 3)])
def test_sumnorm_unit_sum(fm, nu):
    x = np.random.default_rng(7).standard_normal((50, 16)).astype(np.float32)
    f = oracle.features(x, fm, nu, True)
    assert np.allclose(f.sum(-1), 1.0, atol=1e-14) and (f >= 0).all()


def test_feature_dims():
    assert oracle.feature_dim("elu1", 64) == 64
    assert oracle.feature_dim("dpfp", 64, 1) == 128
    assert oracle.feature_dim("dpfp", 64, 3) == 384
    assert oracle.feature_dim("poly2", 16) == 256
    assert oracle.feature_dim("dpfp", 4, 8) == 0      # nu must stay below 2D


# ------------------------------------------------------------------ sequences

@pytest.mark.parametrize("case", _golden()["sequences"], ids=lambda c: c["name"])
def test_golden_sequences(case):
    q = np.array(case["q"], np.float32)[None]
    k = np.array(case["k"], np.float32)[None]
    v = np.array(case["v"], np.float32)[None]
    want = np.array([[_ev(e) for e in row] for row in case["out"]])
    if case["causal"]:
        beta = np.array(case["beta"], np.float32)[None] if "beta" in case else None
        got = oracle.variant_causal(q, k, v, case["fm"], case["nu"], case["norm"], case["update"], beta=beta)[0][0]
    else:
        got = oracle.variant_noncausal(q, k, v, case["fm"], case["nu"], case["norm"])[0]
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13), (got, want)


# DPFP is paired with sum normalisation or none: with the denominator of TaR
# eq. (12) a query whose adjacent sign pairs match no key seen so far has a
# zero denominator (about one first row in eight at D = 16).
VARIANTS = [("elu1", 1, "den"), ("elu1", 1, "sum"), ("elu1", 1, "none"), ("dpfp", 1, "sum"),
            ("dpfp", 2, "sum"), ("dpfp", 3, "none"), ("poly2", 1, "den"), ("poly2", 1, "none")]


@pytest.mark.parametrize("fm,nu,norm", VARIANTS)
def test_sum_update_equals_definition(fm, nu, norm):
    D = 8 if fm == "poly2" else 16
    q, k, v, _ = _rand(3, 37, D, 5, seed=11, scale=0.7)
    out, _, _ = oracle.variant_causal(q, k, v, fm, nu, norm)
    ref = definition_variant(q, k, v, fm, nu, norm, causal=True)
    assert _rel(out, ref) <= 1e-11
    outn = oracle.variant_noncausal(q, k, v, fm, nu, norm)
    refn = definition_variant(q, k, v, fm, nu, norm, causal=False)
    assert _rel(outn, refn) <= 1e-11


def test_elu1_den_matches_base_oracle():
    q, k, v, _ = _rand(2, 50, 16, 8, seed=12)
    a = oracle.variant_causal(q, k, v, "elu1", 1, "den")
    b = oracle.causal(q, k, v)
    for x, y in zip(a, b):
        assert _rel(x, y) <= 1e-13


def delta_ut(q, k, v, beta, S0, fm, nu, C):
    """Delta rule evaluated chunk by chunk, independent of the token loop.

    With unit-free pseudo-values u_t = beta_t (v_t - S_{t-1}^T k_t) the state is
    S_t = S_0 + sum_{s<=t} k_s u_s^T inside a chunk, so
        u_t = beta_t (v_t - S_0^T k_t - sum_{s<t} (k_s . k_t) u_s),
    i.e. (I + diag(beta) tril(K K^T, -1)) U = diag(beta) (V - K S_0): a unit
    lower-triangular system solved here with numpy.  Then
        Y = Q S_0 + tril(Q K^T) U  (read-out after each token's update),
        S_C = S_0 + K^T U.
    """
    Kf = features_np(k, fm, nu, True)
    Qf = features_np(q, fm, nu, True)
    v = v.astype(np.float64)
    beta = beta.astype(np.float64)
    S = S0.copy()
    outs = []
    for c0 in range(0, len(Kf), C):
        K, Q, V, b = Kf[c0:c0 + C], Qf[c0:c0 + C], v[c0:c0 + C], beta[c0:c0 + C]
        n = len(K)
        A = np.eye(n) + b[:, None] * np.tril(K @ K.T, -1)
        U = np.linalg.solve(A, b[:, None] * (V - K @ S))
        outs.append(Q @ S + np.tril(Q @ K.T) @ U)
        S = S + K.T @ U
    return np.concatenate(outs), S


@pytest.mark.parametrize("fm,nu,D,C", [("elu1", 1, 16, 8), ("elu1", 1, 16, 64), ("dpfp", 1, 8, 5), ("dpfp", 2, 8, 16)])
def test_delta_recurrence_equals_chunked(fm, nu, D, C):
    q, k, v, beta = _rand(2, 45, D, 6, seed=13)
    F = oracle.feature_dim(fm, D, nu)
    S0 = np.random.default_rng(14).standard_normal((2, F, 6))
    out, S, _ = oracle.variant_causal(q, k, v, fm, nu, "sum", "delta", beta=beta, S0=S0)
    for h in range(2):
        ro, rS = delta_ut(q[h], k[h], v[h], beta[h], S0[h], fm, nu, C)
        assert _rel(out[h], ro) <= 1e-11
        assert _rel(S[h], rS) <= 1e-11


def test_delta_beta_zero_keeps_state():
    q, k, v, _ = _rand(2, 20, 16, 4, seed=15)
    S0 = np.random.default_rng(16).standard_normal((2, 16, 4))
    out, S, _ = oracle.variant_causal(q, k, v, "elu1", 1, "sum", "delta",
                                      beta=np.zeros((2, 20), np.float32), S0=S0)
    assert np.array_equal(S, S0)
    assert _rel(out, features_np(q, "elu1", 1, True) @ S0) <= 1e-14


def test_delta_one_hot_overwrite():
    """beta = 1 on one-hot keys (DPFP-1, D = 2, sum-normalised) replaces the
    key's slot, so a query in the same quadrant reads the newest value."""
    rng = np.random.default_rng(17)
    N = 64
    k = rng.standard_normal((1, N, 2)).astype(np.float32)
    q = k.copy()                                   # query the key just written
    v = rng.standard_normal((1, N, 3)).astype(np.float32)
    out, S, _ = oracle.variant_causal(q, k, v, "dpfp", 1, "sum", "delta", beta=np.ones((1, N), np.float32))
    assert np.allclose(out[0], v[0], atol=1e-13)
    last = {}
    quad = np.where(k[0, :, 0] > 0, np.where(k[0, :, 1] > 0, 0, 3), np.where(k[0, :, 1] > 0, 1, 2))
    for t in range(N):
        last[int(quad[t])] = v[0, t]
    for slot in range(4):
        want = last.get(slot, np.zeros(3))
        assert np.allclose(S[0, slot], want, atol=1e-13)


@pytest.mark.parametrize("update,norm,fm", [("delta", "sum", "dpfp"), ("sum", "den", "elu1"), ("sum", "none", "dpfp")])
def test_split_carry_equals_whole(update, norm, fm):
    q, k, v, beta = _rand(2, 40, 8, 4, seed=18)
    nu = 1
    whole, Sw, zw = oracle.variant_causal(q, k, v, fm, nu, norm, update, beta=beta)
    a, Sa, za = oracle.variant_causal(q[:, :17], k[:, :17], v[:, :17], fm, nu, norm, update, beta=beta[:, :17])
    b, Sb, zb = oracle.variant_causal(q[:, 17:], k[:, 17:], v[:, 17:], fm, nu, norm, update, beta=beta[:, 17:],
                                      S0=Sa, z0=za if norm == "den" else None)
    assert _rel(np.concatenate([a, b], 1), whole) <= 1e-12
    assert _rel(Sb, Sw) <= 1e-12


# ------------------------------------------------------------------ planted mistakes

def _pins_pass(mutant):
    """True if every pin below still holds with the planted mistake."""
    g = _golden()
    ok = True
    for case in g["sequences"]:
        if not case["causal"]:
            continue
        q = np.array(case["q"], np.float32)[None]
        k = np.array(case["k"], np.float32)[None]
        v = np.array(case["v"], np.float32)[None]
        beta = np.array(case["beta"], np.float32)[None] if "beta" in case else None
        want = np.array([[_ev(e) for e in row] for row in case["out"]])
        got = oracle.variant_causal(q, k, v, case["fm"], case["nu"], case["norm"], case["update"],
                                    beta=beta, mutant=mutant)[0][0]
        ok &= bool(np.allclose(got, want, rtol=1e-12, atol=1e-12))
    for fm, nu, norm in VARIANTS:
        D = 8 if fm == "poly2" else 16
        q, k, v, _ = _rand(2, 21, D, 3, seed=19, scale=0.7)
        out = oracle.variant_causal(q, k, v, fm, nu, norm, mutant=mutant)[0]
        ok &= _rel(out, definition_variant(q, k, v, fm, nu, norm, causal=True)) <= 1e-10
    for fm, nu, D in [("elu1", 1, 16), ("dpfp", 1, 8)]:
        q, k, v, beta = _rand(1, 30, D, 4, seed=20)
        F = oracle.feature_dim(fm, D, nu)
        out, S, _ = oracle.variant_causal(q, k, v, fm, nu, "sum", "delta", beta=beta, mutant=mutant)
        ro, rS = delta_ut(q[0], k[0], v[0], beta[0], np.zeros((F, 4)), fm, nu, 8)
        ok &= _rel(out[0], ro) <= 1e-10 and _rel(S[0], rS) <= 1e-10
    return ok


def test_pins_accept_the_oracle():
    assert _pins_pass(0)


@pytest.mark.parametrize("name", sorted(oracle.VARIANT_MUTANTS))
def test_planted_mistake_caught(name):
    assert not _pins_pass(oracle.VARIANT_MUTANTS[name]), name
