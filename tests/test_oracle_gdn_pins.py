"""Pins of the oracle's Gated DeltaNet values (u of the gated delta rule), none of which
reuses its code.

* The gated delta rule written as a matrix recurrence with dense numpy products,
  S_t = a_t S_{t-1} (I - beta_t k_t k_tᵀ) + beta_t v_t k_tᵀ and o_t = S_t q_t, equals the
  masked form with the transformed values and lambda = 1 (the attention form of the
  model), for grouped and ungrouped heads.
* beta = 0 gives u = 0.
* Orthonormal keys, each seen once: S_{t-1} k_t = 0, so u_t = beta_t v_t.
"""
import numpy as np
import pytest

from oracle import oracle


def _inputs(rng, B, T, H, hpg, dk, dv):
    G = H // hpg
    q = rng.standard_normal((B, T, G, dk))
    k = rng.standard_normal((B, T, G, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    a = rng.uniform(0.5, 1.0, (B, T, H))
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    return q, k, v, a, beta


@pytest.mark.parametrize("T,H,hpg", [(1, 1, 1), (13, 2, 2), (40, 3, 1)])
def test_attention_form_equals_matrix_recurrence(T, H, hpg):
    rng = np.random.default_rng(40 + T)
    dk, dv = 6, 4
    q, k, v, a, beta = _inputs(rng, 2, T, H, hpg, dk, dv)
    L = max(1, (T - 1).bit_length() + 1)
    o = oracle.gdn_forward(q, k, v, a, beta, np.ones((2, T, H, L)))
    G = H // hpg
    for b in range(2):
        for h in range(H):
            g = h // hpg
            S = np.zeros((dv, dk))
            for t in range(T):
                kt = k[b, t, g]
                S = a[b, t, h] * S @ (np.eye(dk) - beta[b, t, h] * np.outer(kt, kt)) \
                    + beta[b, t, h] * np.outer(v[b, t, h], kt)
                np.testing.assert_allclose(o[b, t, h], S @ q[b, t, g], rtol=1e-10, atol=1e-12)
    assert G >= 1


def test_zero_beta_gives_zero_values():
    rng = np.random.default_rng(3)
    q, k, v, a, beta = _inputs(rng, 1, 20, 2, 1, 5, 3)
    assert np.all(oracle.gdn_values(k, v, a, np.zeros_like(beta)) == 0.0)


def test_orthonormal_keys_pass_values_through():
    rng = np.random.default_rng(4)
    T = dk = 8
    k = np.eye(dk)[None, :, None, :]          # k_t = e_t
    v = rng.standard_normal((1, T, 1, 3))
    a = rng.uniform(0.3, 1.0, (1, T, 1))
    beta = rng.uniform(0.0, 1.0, (1, T, 1))
    u = oracle.gdn_values(k, v, a, beta)
    np.testing.assert_allclose(u, beta[..., None] * v, rtol=1e-14, atol=1e-14)
