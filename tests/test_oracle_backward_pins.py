"""Pins of the oracle's backward (gradients of sum(dO * o)), none of which reuses its code.

* Central finite differences of the forward oracle (Form Q), element by element, on tiny
  inputs: a dropped term, a wrong sign or a wrong index in any gradient fails here.
* Euler's identity: o_t is linear in the lambda_t vector, so
  sum_l lambda_t^l dlambda_t^l = dO_t . o_t for every (t, h).
* The linear-attention special case (lambda = 1, a = 1): the gradients of
  o = tril(Q Kᵀ) V written with dense matrices.
"""
import numpy as np
import pytest

from oracle import oracle


def _inputs(rng, B, T, H, hpg, dk, dv, L):
    G = H // hpg
    q = rng.standard_normal((B, T, G, dk))
    k = rng.standard_normal((B, T, G, dk))
    v = rng.standard_normal((B, T, H, dv))
    a = rng.uniform(0.3, 1.0, (B, T, H))
    lam = rng.uniform(0.2, 2.0, (B, T, H, L))
    dO = rng.standard_normal((B, T, H, dv))
    return q, k, v, a, lam, dO


def _loss(q, k, v, a, lam, dO):
    return float(np.sum(dO * oracle.form_q(q, k, v, a, lam)))


@pytest.mark.parametrize("T,H,hpg", [(1, 1, 1), (5, 2, 2), (9, 2, 1), (16, 2, 2)])
def test_backward_matches_finite_differences(T, H, hpg):
    rng = np.random.default_rng(100 + T)
    dk, dv = 3, 2
    L = (T - 1).bit_length() + 2  # one level more than T needs: its gradient is zero
    x = list(_inputs(rng, 1, T, H, hpg, dk, dv, L))
    dq, dkk, dvv, dla, dl = oracle.backward(*x)
    grads = [dq, dkk, dvv, dla / x[3], dl]  # the finite differences below move a itself
    eps = 1e-6
    for idx in range(5):  # q, k, v, a, lam
        base = x[idx]
        num = np.zeros_like(base)
        for pos in np.ndindex(base.shape):
            orig = base[pos]
            base[pos] = orig + eps
            fp = _loss(*x)
            base[pos] = orig - eps
            fm = _loss(*x)
            base[pos] = orig
            num[pos] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(grads[idx], num, rtol=1e-6, atol=1e-7,
                                   err_msg=["dq", "dk", "dv", "da", "dlam"][idx])
    assert np.all(grads[4][..., (T - 1).bit_length() + 1:] == 0.0)
    # in log space: a -> a * exp(+-eps) moves log a by +-eps
    num = np.zeros_like(dla)
    a0 = x[3].copy()
    for pos in np.ndindex(a0.shape):
        x[3] = a0.copy()
        x[3][pos] = a0[pos] * np.exp(eps)
        fp = _loss(*x)
        x[3][pos] = a0[pos] * np.exp(-eps)
        fm = _loss(*x)
        num[pos] = (fp - fm) / (2 * eps)
    x[3] = a0
    np.testing.assert_allclose(dla, num, rtol=1e-6, atol=1e-7, err_msg="dloga")


def test_euler_identity_for_lambda():
    rng = np.random.default_rng(7)
    q, k, v, a, lam, dO = _inputs(rng, 2, 37, 4, 2, 8, 4, 7)
    dl = oracle.backward(q, k, v, a, lam, dO)[4]
    o = oracle.form_q(q, k, v, a, lam)
    np.testing.assert_allclose(np.sum(lam * dl, axis=-1), np.sum(dO * o, axis=-1), rtol=1e-10,
                               atol=1e-10)


def test_linear_attention_special_case():
    """lambda = 1, a = 1: o = tril(Q Kᵀ) V per head, so dq = tril(dO Vᵀ) K,
    dk = tril(dO Vᵀ)ᵀ Q, dv = tril(Q Kᵀ)ᵀ dO, and d(log a_r) = sum over t >= r, s < r of
    (q_t . k_s)(dO_t . v_s)."""
    rng = np.random.default_rng(9)
    T, dk, dv, L = 21, 5, 3, 6
    q, k, v, _, _, dO = _inputs(rng, 1, T, 1, 1, dk, dv, L)
    a = np.ones((1, T, 1))
    lam = np.ones((1, T, 1, L))
    dq, dkk, dvv, dla, _ = oracle.backward(q, k, v, a, lam, dO)
    Q, K, V, D = q[0, :, 0], k[0, :, 0], v[0, :, 0], dO[0, :, 0]
    mask = np.tril(np.ones((T, T)))
    P = mask * (Q @ K.T)
    dP = mask * (D @ V.T)
    np.testing.assert_allclose(dq[0, :, 0], dP @ K, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dkk[0, :, 0], dP.T @ Q, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dvv[0, :, 0], P.T @ D, rtol=1e-12, atol=1e-12)
    A = P * (D @ V.T)
    want = np.array([A[r:, :r].sum() for r in range(T)])
    np.testing.assert_allclose(dla[0, :, 0], want, rtol=1e-12, atol=1e-12)
