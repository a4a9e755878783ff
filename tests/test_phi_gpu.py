"""The device feature map phi(x) = elu(x) + 1 ("Transformers are RNNs",
sec. 3.2.1 eq. (7)) of the tensor-core kernels, pinned value by value.

The tensor-core kernels apply phi to Q and K tiles in shared memory and never
store the result, so the tests read it back through outputs that expose it
exactly:

* keys: a causal call with V = identity (v_j = e_j) and a zero start state
  leaves S[d][j] = phi(K[j][d]) in its fp32 final state (one product with
  1.0 per entry, no rounding), so the state holds the bf16 feature values the
  kernel computed, for 4096 (D = 64) or 16384 (D = 128) inputs spanning
  [-20, 5];
* queries: unit keys phi(k_j) = e_j (zero on the diagonal, -100 elsewhere,
  whose phi underflows to 0) and V = identity make output row i equal to
  phi(q_i) / sum_d phi(q_i)_d.  A row holding 0, 1, -1 and -100 gives
  outputs fixed exactly by phi(0) = 1, phi(1) = 2 and phi(-1) = e^-1; rows of
  other values give phi(q_m) / phi(q_0) = out_m / out_0 with q_0 = 0.

The device evaluates phi in fp32 and rounds to bf16 once, so each key feature
must be the correctly rounded value of the fp64 phi (within a 2^-10 fraction
of an ulp, for the exponential's own error); the query ratios carry two more
bf16 output roundings.
"""
import numpy as np
import pytest
import torch

import oracle
from weight_recurrence_gb300 import la

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.lib()
    oracle.build()


def _grid(n):
    """n bf16 inputs spanning [-20, 5], with the spot values 0, 1, -1 first."""
    spots = torch.tensor([0.0, 1.0, -1.0, -4.5, 5.0, -20.0, -0.0, 2.0 ** -10])
    x = torch.linspace(-20.0, 5.0, n - len(spots))
    return torch.cat([spots, x]).to(torch.bfloat16)


def _half_ulp_bf16(y):
    """Half a bf16 ulp at |y| (y > 0, normal)."""
    e = np.floor(np.log2(np.abs(y)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def _phi64(x):
    return oracle.phi_np(np.asarray(x, np.float64))


@pytest.mark.parametrize("D", [64, 128])
def test_key_features_are_correctly_rounded(D):
    """S[d][j] = phi(K[j][d]) exactly, from the causal kernel's final state."""
    x = _grid(D * D)
    k = x.reshape(1, 1, D, D)                          # K[j][d] = x[j * D + d]
    v = torch.eye(D, dtype=torch.bfloat16).reshape(1, 1, D, D)
    q = torch.zeros_like(k)
    S = torch.zeros(1, 1, D, D, device=DEV)
    z = torch.zeros(1, 1, D, device=DEV)
    la.la_forward_causal(q.to(DEV), k.to(DEV), v.to(DEV), S=S, z=z, want_out=False)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    dev_phi = S[0, 0].cpu().double().numpy().T.reshape(-1)     # [j][d] order = x order
    ref = _phi64(x.double().numpy())
    err = np.abs(dev_phi - ref)
    bound = _half_ulp_bf16(ref) * (1.0 + 2.0 ** -10)
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), (float(x[worst]), dev_phi[worst], ref[worst])
    # spot values: phi(0) = 1, phi(1) = 2, phi(-1) = e^-1 rounded to bf16
    assert dev_phi[0] == 1.0 and dev_phi[1] == 2.0
    assert dev_phi[2] == float(torch.tensor(np.exp(-1.0), dtype=torch.float32).to(torch.bfloat16))
    # z = sum_j phi(K[j]) over the same values (fp32 accumulation)
    zref = dev_phi.reshape(D, D).sum(axis=0)
    assert np.allclose(z[0, 0].cpu().double().numpy(), zref, rtol=1e-5, atol=0)


def _query_probe(D, nq, causal):
    """Inputs whose output rows reveal phi of the query rows (see the module
    docstring); returns q, k, v and the index of the first probe row."""
    first = D if causal else 0               # causal: probe rows see every unit key
    N = first + nq
    if not causal:
        N = max(N, D)
    k = torch.full((N, D), -100.0)
    k[:D, :D] = torch.where(torch.eye(D) > 0, torch.zeros(D, D), torch.full((D, D), -100.0))
    v = torch.zeros(N, D)
    v[:D] = torch.eye(D)
    q = torch.zeros(N, D)
    x = _grid(nq * (D - 1)).float().reshape(nq, D - 1)
    q[first:first + nq, 1:] = x
    spot = torch.full((D,), -100.0)
    spot[:3] = torch.tensor([0.0, 1.0, -1.0])
    q[first] = spot                          # exact spot rows, first and last
    q[first + nq - 1] = spot
    as_in = lambda t: t.to(torch.bfloat16).reshape(1, 1, N, D)  # noqa: E731
    return as_in(q), as_in(k), as_in(v), first


def _expected_spot_row(D):
    """Output of the spot row in fp32 arithmetic as the kernels form it:
    den = 1 + 2 + bf16(e^-1), inv = 1 / den, out_m = bf16(phi_m * inv)."""
    p = np.zeros(D, np.float32)
    p[0], p[1] = 1.0, 2.0
    p[2] = float(torch.tensor(np.exp(-1.0), dtype=torch.float32).to(torch.bfloat16))
    den = np.float32(p[0] + p[1] + p[2])
    inv = np.float32(1.0) / den
    return torch.from_numpy((p * inv).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("form,D", [("noncausal", 64), ("noncausal", 128), ("causal", 64), ("causal", 128)])
def test_query_features(form, D):
    nq = 128
    q, k, v, first = _query_probe(D, nq, form == "causal")
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    if form == "causal":
        out = la.la_forward_causal(qd, kd, vd)
    else:
        out = la.la_forward_noncausal(qd, kd, vd)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    out = out[0, 0].cpu()
    # the spot rows, exactly
    for r in (first, first + nq - 1):
        assert torch.equal(out[r], _expected_spot_row(D)), (r, out[r, :4])
    # the other rows: phi(q_m) = out_m / out_0 (q_0 = 0), two output roundings
    o = out[first + 1:first + nq - 1].double().numpy()
    x = q[0, 0, first + 1:first + nq - 1, 1:].double().numpy()
    meas = o[:, 1:] / o[:, :1]
    ref = _phi64(x)
    rel = np.abs(meas / ref - 1.0)
    worst = np.unravel_index(int(np.argmax(rel)), rel.shape)
    assert rel.max() <= 3.0 * 2.0 ** -8 + 2.0 ** -12, (float(x[worst]), meas[worst], ref[worst])
