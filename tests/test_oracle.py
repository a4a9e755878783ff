"""Pins for the fp64 oracle, checked against things other than the oracle itself.

Sources ("Transformers are RNNs", read in its Chinese translation):
  * hand-worked fixtures in tests/golden/hand_examples.json (eqs. (3), (4), (7), (8));
  * the definition form (numpy quadratic form of eqs. (3)/(4)/(8)) vs the C
    recurrence of eqs. (10)-(12)/(16)-(20) - two independent programs;
  * a literal pure-Python triple loop of eq. (3) on tiny inputs;
  * closed forms: constant V reproduces itself (the non-negative similarity of
    sec. 3.2 makes every output a convex combination of value rows), equal keys
    give prefix means; invariants: prefix independence (sec. 3.3), state carry
    (sec. 3.3.2), affine equivariance in V, last causal row = non-causal row.
  * planted mistakes in the C oracle must each break at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import definition_causal, definition_noncausal, definition_rows, phi_np
from weight_recurrence_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
E = math.exp(-1.0)


def _ev(expr):
    return float(eval(expr, {"E": E, "math": math}))


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(shape_qk, M, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal(shape_qk) * scale).astype(np.float32)
    k = (rng.standard_normal(shape_qk) * scale).astype(np.float32)
    v = rng.standard_normal(shape_qk[:-1] + (M,)).astype(np.float32)
    return q, k, v


def _loop_bruteforce(q, k, v, causal):
    """eq. (3) written out as plain loops: sim(q,k) = sum_d phi(q_d) phi(k_d)."""
    N, D = q.shape
    M = v.shape[1]

    def phi(x):
        return x + 1.0 if x > 0 else math.exp(x)

    out = [[0.0] * M for _ in range(N)]
    for i in range(N):
        num = [0.0] * M
        den = 0.0
        for j in range(N):
            if causal and j > i:
                continue
            s = 0.0
            for d in range(D):
                s += phi(float(q[i, d])) * phi(float(k[j, d]))
            den += s
            for m in range(M):
                num[m] += s * float(v[j, m])
        for m in range(M):
            out[i][m] = num[m] / den
    return np.array(out)


# ----------------------------------------------------------------- fixtures

def test_phi_golden(oracle_mod):
    g = _golden()["phi"]["cases"]
    for x, y in g:
        assert oracle_mod.phi(_ev(x)) == pytest.approx(_ev(y), rel=1e-15, abs=0)
        assert float(phi_np(_ev(x))) == pytest.approx(_ev(y), rel=1e-15, abs=0)


def test_phi_positive_and_continuous(oracle_mod):
    xs = np.linspace(-30, 30, 2001)
    vals = np.array([oracle_mod.phi(x) for x in xs])
    assert np.all(vals > 0)
    assert np.all(np.diff(vals) > 0)          # strictly increasing
    assert oracle_mod.phi(-1e-12) == pytest.approx(1.0, abs=1e-11)
    assert oracle_mod.phi(1e-12) == pytest.approx(1.0, abs=1e-11)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_hand_examples(oracle_mod, idx):
    ex = _golden()["examples"][idx]
    q = np.array(ex["q"], np.float32)
    k = np.array(ex["k"], np.float32)
    v = np.array(ex["v"], np.float32)
    want_c = np.array([[_ev(e) for e in row] for row in ex["causal"]])
    want_n = np.array([[_ev(e) for e in row] for row in ex["noncausal"]])
    out_c, _, _ = oracle_mod.causal(q[None], k[None], v[None])
    out_n, _, _ = oracle_mod.noncausal(q[None], k[None], v[None])
    np.testing.assert_allclose(out_c[0], want_c, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out_n[0], want_n, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(definition_causal(q, k, v), want_c, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(definition_noncausal(q, k, v), want_n, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(_loop_bruteforce(q, k, v, True), want_c, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(_loop_bruteforce(q, k, v, False), want_n, rtol=1e-14, atol=1e-15)


def test_decode_golden(oracle_mod):
    ex = _golden()["examples"][0]
    q = np.array(ex["q"], np.float32)
    k = np.array(ex["k"], np.float32)
    v = np.array(ex["v"], np.float32)
    S = np.zeros((1, 1, 1), np.float64)
    z = np.zeros((1, 1), np.float64)
    y0 = oracle_mod.decode_step(q[0][None], k[0][None], v[0][None], S, z)
    y1 = oracle_mod.decode_step(q[1][None], k[1][None], v[1][None], S, z)
    assert y0[0, 0] == pytest.approx(1.0, rel=1e-15)        # first step returns v
    assert y1[0, 0] == pytest.approx(_ev(ex["causal"][1][0]), rel=1e-15)


# ------------------------------------------------- independent forms agree

@pytest.mark.parametrize("N,D,M,scale", [(1, 4, 3, 1.0), (37, 8, 5, 1.0), (130, 16, 16, 0.25), (64, 32, 8, 3.0)])
def test_recurrence_equals_definition(oracle_mod, N, D, M, scale):
    q, k, v = _rand((2, 3, N, D), M, seed=N * 7 + D, scale=scale)
    out_c, S, z = oracle_mod.causal(q, k, v)
    ref_c = definition_causal(q, k, v)
    np.testing.assert_allclose(out_c, ref_c, rtol=1e-12, atol=1e-12)
    out_n, kv, ks = oracle_mod.noncausal(q, k, v)
    np.testing.assert_allclose(out_n, definition_noncausal(q, k, v), rtol=1e-12, atol=1e-12)
    # the non-causal summaries equal the final causal state (both are sums over all j)
    np.testing.assert_allclose(kv, S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ks, z, rtol=1e-12, atol=1e-12)


def test_pure_python_loops(oracle_mod):
    q, k, v = _rand((6, 3), 2, seed=5)
    out_c, _, _ = oracle_mod.causal(q[None], k[None], v[None])
    out_n, _, _ = oracle_mod.noncausal(q[None], k[None], v[None])
    np.testing.assert_allclose(out_c[0], _loop_bruteforce(q, k, v, True), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(out_n[0], _loop_bruteforce(q, k, v, False), rtol=1e-13, atol=1e-14)


def test_sampled_rows_match_full():
    q, k, v = _rand((200, 8), 4, seed=11)
    rows = np.array([0, 1, 63, 64, 65, 199])
    np.testing.assert_allclose(definition_rows(q, k, v, rows, True), definition_causal(q, k, v)[rows],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(definition_rows(q, k, v, rows, False), definition_noncausal(q, k, v)[rows],
                               rtol=1e-12, atol=1e-13)


# --------------------------------------------------- closed forms/invariants

def test_last_causal_row_is_noncausal(oracle_mod):
    q, k, v = _rand((2, 2, 50, 8), 6, seed=3)
    out_c, _, _ = oracle_mod.causal(q, k, v)
    out_n, _, _ = oracle_mod.noncausal(q, k, v)
    np.testing.assert_allclose(out_c[..., -1, :], out_n[..., -1, :], rtol=1e-13, atol=1e-14)


def test_constant_v_reproduces_itself(oracle_mod):
    q, k, _ = _rand((1, 3, 40, 8), 5, seed=4, scale=2.0)
    c = np.array([1.5, -2.25, 0.0, 7.0, -0.125], np.float32)
    v = np.broadcast_to(c, (1, 3, 40, 5)).copy()
    for out in (oracle_mod.causal(q, k, v)[0], oracle_mod.noncausal(q, k, v)[0]):
        np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=1e-13, atol=1e-13)


def test_outputs_in_convex_hull(oracle_mod):
    q, k, v = _rand((1, 2, 60, 8), 4, seed=9)
    out, _, _ = oracle_mod.causal(q, k, v)
    v64 = v.astype(np.float64)
    for i in range(60):
        lo = v64[..., : i + 1, :].min(axis=-2)
        hi = v64[..., : i + 1, :].max(axis=-2)
        assert np.all(out[..., i, :] >= lo - 1e-12) and np.all(out[..., i, :] <= hi + 1e-12)


def test_equal_keys_give_prefix_mean(oracle_mod):
    rng = np.random.default_rng(12)
    N, D, M = 33, 6, 3
    q = rng.standard_normal((1, N, D)).astype(np.float32)
    k = np.broadcast_to(rng.standard_normal(D).astype(np.float32), (1, N, D)).copy()
    v = rng.standard_normal((1, N, M)).astype(np.float32)
    out_c, _, _ = oracle_mod.causal(q, k, v)
    want = np.cumsum(v[0].astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(out_c[0], want, rtol=1e-12, atol=1e-13)
    out_n, _, _ = oracle_mod.noncausal(q, k, v)
    np.testing.assert_allclose(out_n[0], np.broadcast_to(v[0].astype(np.float64).mean(0), (N, M)),
                               rtol=1e-12, atol=1e-13)


def test_prefix_independence(oracle_mod):
    q, k, v = _rand((1, 1, 80, 8), 8, seed=21)
    out1, _, _ = oracle_mod.causal(q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[..., 50:, :] += 1.0
    k2[..., 50:, :] -= 2.0
    v2[..., 50:, :] *= 3.0
    out2, _, _ = oracle_mod.causal(q2, k2, v2)
    np.testing.assert_array_equal(out1[..., :50, :], out2[..., :50, :])
    assert not np.allclose(out1[..., 50:, :], out2[..., 50:, :])


@pytest.mark.parametrize("split", [1, 17, 64, 99])
def test_state_carry(oracle_mod, split):
    q, k, v = _rand((2, 1, 100, 8), 8, seed=31)
    full, S, z = oracle_mod.causal(q, k, v)
    a, S1, z1 = oracle_mod.causal(q[..., :split, :], k[..., :split, :], v[..., :split, :])
    b, S2, z2 = oracle_mod.causal(q[..., split:, :], k[..., split:, :], v[..., split:, :], S0=S1, z0=z1)
    np.testing.assert_allclose(np.concatenate([a, b], axis=-2), full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(z2, z, rtol=1e-12, atol=1e-12)
    # the sampled-row definition form agrees with a carried-in prefix state
    rows = np.unique(np.array([0, min(5, 99 - split), 99 - split]))
    got = definition_rows(q[0, 0, split:], k[0, 0, split:], v[0, 0, split:], rows, True,
                          prefix_state=(S1[0, 0], z1[0, 0]))
    np.testing.assert_allclose(got, full[0, 0, split:][rows], rtol=1e-12, atol=1e-13)


def test_affine_equivariance_in_v(oracle_mod):
    q, k, v = _rand((1, 2, 45, 8), 4, seed=41)
    a, b = np.float32(-2.5), np.float32(0.75)
    out, _, _ = oracle_mod.causal(q, k, v)
    out2, _, _ = oracle_mod.causal(q, k, (a * v + b).astype(np.float32))
    # a*v+b is rounded to fp32 on input, hence the 1e-6 bound
    np.testing.assert_allclose(out2, a * out + b, rtol=1e-6, atol=1e-6)


def test_decode_matches_causal(oracle_mod):
    q, k, v = _rand((2, 3, 20, 8), 8, seed=51)
    out, S, z = oracle_mod.causal(q, k, v)
    Sd = np.zeros((2, 3, 8, 8))
    zd = np.zeros((2, 3, 8))
    for t in range(20):
        y = oracle_mod.decode_step(q[..., t, :], k[..., t, :], v[..., t, :], Sd, zd)
        np.testing.assert_allclose(y, out[..., t, :], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(Sd, S, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(zd, z, rtol=1e-13, atol=1e-13)


def test_seeded_inputs_are_deterministic():
    a = inputs.qkv(1, 2, 10, 16, 16, seed=7)
    b = inputs.qkv(1, 2, 10, 16, 16, seed=7)
    for x, y in zip(a, b):
        assert (x.float() == y.float()).all()


# ------------------------------------------------------- planted mistakes

def _pins_pass(oracle_mod, mutant):
    """Run the pin checks against an oracle with a planted mistake; True if all pass."""
    try:
        for ex in _golden()["examples"]:
            q = np.array(ex["q"], np.float32)[None]
            k = np.array(ex["k"], np.float32)[None]
            v = np.array(ex["v"], np.float32)[None]
            want_c = np.array([[_ev(e) for e in row] for row in ex["causal"]])
            want_n = np.array([[_ev(e) for e in row] for row in ex["noncausal"]])
            np.testing.assert_allclose(oracle_mod.causal(q, k, v, mutant=mutant)[0][0], want_c, rtol=1e-12)
            np.testing.assert_allclose(oracle_mod.noncausal(q, k, v, mutant=mutant)[0][0], want_n, rtol=1e-12)
        q, k, v = _rand((1, 2, 30, 8), 8, seed=77)
        np.testing.assert_allclose(oracle_mod.causal(q, k, v, mutant=mutant)[0], definition_causal(q, k, v),
                                   rtol=1e-10)
        np.testing.assert_allclose(oracle_mod.noncausal(q, k, v, mutant=mutant)[0],
                                   definition_noncausal(q, k, v), rtol=1e-10)
        return True
    except (AssertionError, FloatingPointError, ValueError):
        return False


@pytest.mark.parametrize("name", ["relu", "no_z_update", "read_before_update", "transpose_S",
                                  "phi_sign", "shifted_v", "den_uses_k"])
def test_planted_mistake_is_caught(oracle_mod, name):
    assert _pins_pass(oracle_mod, 0)
    with np.errstate(all="ignore"):
        assert not _pins_pass(oracle_mod, oracle_mod.MUTANTS[name]), name
