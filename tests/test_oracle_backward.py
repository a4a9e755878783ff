"""Pins for the backward oracle, checked against things other than the oracle.

The pages state that the gradient of the causal form is a cumulative sum
computable in constant extra memory ("Transformers are RNNs" sec. 3.3.1), but
print neither its equations (13)-(15) nor Algorithm 1.  The oracle therefore
applies the chain rule to eqs. (10)-(12); these tests pin it with:
  * central finite differences of the definition form (eqs. (3), (4), (8),
    numpy fp64) - an independent program - on tiny inputs;
  * torch autograd of the definition form in fp64 on medium inputs;
  * closed forms: a constant V makes every output constant, so dQ = dK = 0;
  * chaining: the backward of a split sequence, joined through the state
    gradients dS_0 / dZ_0, equals the backward of the whole sequence;
  * finite differences in the carried-in state (dS_0, dZ_0);
  * every planted mistake fails at least one of these.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import definition_causal, definition_noncausal


def _rand(seed, shape, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def _case(seed, B, N, D, M, scale=1.0):
    return (_rand(seed, (B, N, D), scale), _rand(seed + 1, (B, N, D), scale),
            _rand(seed + 2, (B, N, M)), _rand(seed + 3, (B, N, M)))


def _loss(defn, q, k, v, G):
    return float((defn(q, k, v) * np.asarray(G, np.float64)).sum())


def _fd_grads(defn, q, k, v, G, h=1e-6):
    """Central differences of L = sum(G * O_def) in every input element (fp64)."""
    out = []
    base = [np.asarray(a, np.float64) for a in (q, k, v)]
    for which in range(3):
        g = np.zeros_like(base[which])
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p = [a.copy() for a in base]
            args_m = [a.copy() for a in base]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            g[idx] = (_loss(defn, *args_p, G) - _loss(defn, *args_m, G)) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed,N,D,M", [(10, 5, 3, 2), (20, 7, 2, 3), (30, 1, 4, 2)])
def test_backward_matches_finite_differences(oracle_mod, causal, seed, N, D, M):
    q, k, v, G = _case(seed, 2, N, D, M)
    if causal:
        dq, dk, dv, _, _ = oracle.causal_backward(q, k, v, G)
        fd = _fd_grads(definition_causal, q, k, v, G)
    else:
        dq, dk, dv = oracle.noncausal_backward(q, k, v, G)
        fd = _fd_grads(definition_noncausal, q, k, v, G)
    for got, ref in zip((dq, dk, dv), fd):
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-8)


def _torch_definition(q, k, v, causal):
    fq = torch.where(q > 0, q + 1, torch.exp(torch.clamp(q, max=0.0)))
    fk = torch.where(k > 0, k + 1, torch.exp(torch.clamp(k, max=0.0)))
    w = fq @ fk.transpose(-1, -2)
    if causal:
        N = q.shape[-2]
        w = w * torch.tril(torch.ones(N, N, dtype=w.dtype))
    return (w @ v) / w.sum(-1, keepdim=True)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed,B,N,D,M,scale", [(40, 2, 40, 8, 6, 1.0), (50, 1, 70, 16, 16, 0.5),
                                                (60, 3, 33, 4, 12, 2.0)])
def test_backward_matches_autograd(oracle_mod, causal, seed, B, N, D, M, scale):
    q, k, v, G = _case(seed, B, N, D, M, scale)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    (_torch_definition(tq, tk, tv, causal) * torch.tensor(G, dtype=torch.float64)).sum().backward()
    if causal:
        got = oracle.causal_backward(q, k, v, G)[:3]
    else:
        got = oracle.noncausal_backward(q, k, v, G)
    for g, t in zip(got, (tq, tk, tv)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("causal", [True, False])
def test_constant_v_gives_zero_query_and_key_gradients(oracle_mod, causal):
    q, k, _, G = _case(70, 2, 30, 8, 5)
    v = np.broadcast_to(_rand(74, (2, 1, 5)), (2, 30, 5)).copy()
    res = oracle.causal_backward(q, k, v, G) if causal else oracle.noncausal_backward(q, k, v, G)
    assert np.abs(res[0]).max() < 1e-12 and np.abs(res[1]).max() < 1e-12
    # dV then carries all of G: sum over rows of dV equals sum over rows of G
    np.testing.assert_allclose(res[2].sum(axis=1), np.asarray(G, np.float64).sum(axis=1), rtol=1e-10)


@pytest.mark.parametrize("split", [1, 17, 39])
def test_split_backward_chains_through_state_gradients(oracle_mod, split):
    q, k, v, G = _case(80, 2, 40, 6, 5)
    whole = oracle.causal_backward(q, k, v, G)
    # forward state after the first part, then the second part's backward
    _, S1, z1 = oracle.causal(q[:, :split], k[:, :split], v[:, :split], want_out=False)
    dq2, dk2, dv2, dS1, dz1 = oracle.causal_backward(q[:, split:], k[:, split:], v[:, split:], G[:, split:],
                                                     S0=S1, z0=z1)
    dq1, dk1, dv1, dS0, dz0 = oracle.causal_backward(q[:, :split], k[:, :split], v[:, :split], G[:, :split],
                                                     dSN=dS1, dzN=dz1)
    for part, ref in zip((np.concatenate([dq1, dq2], 1), np.concatenate([dk1, dk2], 1),
                          np.concatenate([dv1, dv2], 1), dS0, dz0), whole):
        np.testing.assert_allclose(part, ref, rtol=1e-10, atol=1e-12)


def test_state_gradients_match_finite_differences(oracle_mod):
    """dS_0, dZ_0 against central differences of the forward oracle in the carried-in state."""
    q, k, v, G = _case(90, 1, 6, 3, 2)
    rng = np.random.default_rng(91)
    S0 = rng.standard_normal((1, 3, 2)) * 2.0
    z0 = np.abs(rng.standard_normal((1, 3))) * 3.0 + 1.0
    _, _, _, dS0, dz0 = oracle.causal_backward(q, k, v, G, S0=S0, z0=z0)
    G64 = np.asarray(G, np.float64)

    def L(S, z):
        out, _, _ = oracle.causal(q, k, v, S0=S, z0=z)
        return float((out * G64).sum())
    h = 1e-6
    for idx in np.ndindex(S0.shape):
        Sp, Sm = S0.copy(), S0.copy()
        Sp[idx] += h
        Sm[idx] -= h
        assert abs((L(Sp, z0) - L(Sm, z0)) / (2 * h) - dS0[idx]) <= 1e-7 * max(1.0, abs(dS0[idx]))
    for idx in np.ndindex(z0.shape):
        zp, zm = z0.copy(), z0.copy()
        zp[idx] += h
        zm[idx] -= h
        assert abs((L(S0, zp) - L(S0, zm)) / (2 * h) - dz0[idx]) <= 1e-7 * max(1.0, abs(dz0[idx]))


@pytest.mark.parametrize("name", ["bwd_no_e", "bwd_dphi_is_phi", "bwd_excl_diag", "bwd_dv_uses_q"])
@pytest.mark.parametrize("causal", [True, False])
def test_planted_backward_mistake_is_caught(oracle_mod, name, causal):
    if not causal and name == "bwd_excl_diag":
        pytest.skip("the non-causal sums have no diagonal to drop")
    q, k, v, G = _case(100, 2, 12, 4, 4)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    (_torch_definition(tq, tk, tv, causal) * torch.tensor(G, dtype=torch.float64)).sum().backward()
    fn = oracle.causal_backward if causal else oracle.noncausal_backward
    got = fn(q, k, v, G, mutant=oracle.MUTANTS[name])[:3]
    worst = max(float(np.abs(g - t.grad.numpy()).max() / (np.abs(t.grad.numpy()).max() + 1e-30))
                for g, t in zip(got, (tq, tk, tv)))
    assert worst > 1e-3, (name, worst)
