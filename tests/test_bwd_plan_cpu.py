"""The algebra of the tensor-core backward pass, checked on the host in fp64.

For plain retention (no feature map, no normaliser) the library computes the
gradients of L = sum_t do_t . o_t + <dS_T, S_T> as three forward passes of the
causal decayed form with the inputs' roles exchanged:

  dQ = forward(queries dO, keys V, values K, initial state S_0^T);
  dV = reversed forward(queries K, keys Q, values dO, initial state dS_T / gamma);
  dK = reversed forward(queries V, keys dO, values Q, initial state dS_T^T / gamma);
  dS_0 = gamma times the dV pass's final state,

where a reversed forward runs over the time-reversed sequences and its output is
reversed back.  This is the chain rule on the recurrence ("Linear attention" page,
"Decoding, training, and what each costs": the gradients are cumulative sums,
forward in time for the queries and backward for the keys and values).  Here
each pass is the brute-force masked form, with an initial state read through
gamma^(t+1), and the result is compared with the oracle's two sweeps.
"""
import numpy as np
import pytest

import oracle


def forward(Q, K, V, gamma, S0):
    """o_t = sum_{s<=t} gamma^(t-s) (q_t . k_s) v_s + gamma^(t+1) q_t S0, and the final
    state gamma^T S0 + sum_s gamma^(T-1-s) k_s^T v_s, for one sequence."""
    T = Q.shape[0]
    n = np.arange(T)
    D = np.where(n[:, None] >= n[None, :], gamma ** np.clip(n[:, None] - n[None, :], 0, None), 0.0)
    O = ((Q @ K.T) * D) @ V + (gamma ** (n + 1))[:, None] * (Q @ S0)
    S = gamma ** T * S0 + (K * (gamma ** (T - 1 - n))[:, None]).T @ V
    return O, S


def reversed_forward(Q, K, V, gamma, S0):
    O, S = forward(Q[::-1], K[::-1], V[::-1], gamma, S0)
    return O[::-1], S


@pytest.mark.parametrize("T,dk,dv,gamma", [(1, 4, 4, 0.9), (37, 8, 5, 0.97), (64, 6, 9, 1.0),
                                           (50, 16, 16, 0.5)])
def test_three_forward_passes_give_the_gradients(T, dk, dv, gamma):
    rng = np.random.default_rng(T * 1000 + dk)
    q, k = rng.standard_normal((2, T, dk))
    v, dO = rng.standard_normal((2, T, dv))
    S0 = rng.standard_normal((dk, dv)) * 0.3
    dST = rng.standard_normal((dk, dv)) * 0.1
    dq, _ = forward(dO, v, k, gamma, S0.T)
    dv_, G0 = reversed_forward(k, q, dO, gamma, dST / gamma)
    dk_, _ = reversed_forward(v, dO, q, gamma, dST.T / gamma)
    dS0 = gamma * G0
    rq, rk, rv, rS0, _ = oracle.recurrent_bwd(q[None, None], k[None, None], v[None, None],
                                              [gamma], dO[None, None], S0=S0[None, None],
                                              dS_T=dST[None, None])
    np.testing.assert_allclose(dq, rq[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk_, rk[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv_, rv[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dS0, rS0[0, 0], rtol=1e-10, atol=1e-12)


def phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


@pytest.mark.parametrize("T,dk,dv,gamma", [(37, 8, 5, 0.97), (64, 6, 9, 1.0)])
def test_three_forward_passes_with_phi(T, dk, dv, gamma):
    """With phi = elu + 1 and no normaliser the same passes run on phi(q), phi(k), and
    the chain rule through phi multiplies the q and k gradients by phi'(x) = 1 above
    zero, e^x at or below."""
    rng = np.random.default_rng(T * 1000 + dk + 1)
    q, k = rng.standard_normal((2, T, dk))
    v, dO = rng.standard_normal((2, T, dv))
    S0 = rng.standard_normal((dk, dv)) * 0.3
    dST = rng.standard_normal((dk, dv)) * 0.1
    qt, kt = phi(q), phi(k)
    dqt, _ = forward(dO, v, kt, gamma, S0.T)
    dv_, G0 = reversed_forward(kt, qt, dO, gamma, dST / gamma)
    dkt, _ = reversed_forward(v, dO, qt, gamma, dST.T / gamma)
    dq = dqt * np.where(q > 0, 1.0, np.exp(np.minimum(q, 0.0)))
    dk_ = dkt * np.where(k > 0, 1.0, np.exp(np.minimum(k, 0.0)))
    rq, rk, rv, rS0, _ = oracle.recurrent_bwd(q[None, None], k[None, None], v[None, None],
                                              [gamma], dO[None, None], S0=S0[None, None],
                                              dS_T=dST[None, None], phi=True)
    np.testing.assert_allclose(dq, rq[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk_, rk[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv_, rv[0, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gamma * G0, rS0[0, 0], rtol=1e-10, atol=1e-12)
