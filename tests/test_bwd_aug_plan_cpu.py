"""The algebra of the normalised backward's tensor-core passes, on the host in fp64.

With phi (elu + 1 or the identity) and the normaliser, n_t = q~_t S_t, u_t = q~_t . z_t,
dd_t = u_t + eps (or max(|u_t|, 1) with the floor) and o_t = n_t / dd_t.  For
L = sum_t do_t . o_t + <dS_T, S_T> + <dz_T, z_T> the gradients with respect to n_t and
u_t are dn_t = do_t / dd_t and du_t = -(do_t . o_t) / dd_t * dd'(u_t).  The library
takes dq, dd and du from the CUDA-core kernel's forward sweep and computes dk and dv
as two forward passes of the plain decayed form over the reversed sequences:

  dk~ = reversed forward(queries [v | 1 | 1], keys [dn | du_hi | du_lo], values q~,
                initial state [dS_T^T; dz_T; 0] / gamma);
  dv  = reversed forward(queries k~, keys q~, values dn, initial state dS_T / gamma);
  dk = dk~ phi'(k), dS_0 = gamma (the dv pass's final state),
  dz_0 = gamma (the sum of the dk~ pass's two extra final-state rows),

with du = du_hi + du_lo (the kernel splits du into two bf16 parts; here any split).
This is the chain rule on the recurrence ("Linear attention" page, "Decoding,
training, and what each costs"); each pass is the brute-force masked form and the
result is compared with the oracle's own backward sweeps.  (dq as a forward pass
over [dn | du] with keys [v | 1 | 1] holds too, and is checked here as well, but the
library does not use it: it is a near-cancellation that bf16 operands do not resolve.)
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


def phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


@pytest.mark.parametrize("phi_on", [True, False], ids=["elu1", "identity"])
@pytest.mark.parametrize("floor", [False, True], ids=["eps", "floor"])
@pytest.mark.parametrize("T,dk,dv,gamma", [(1, 4, 4, 0.9), (37, 6, 5, 0.97), (64, 5, 7, 1.0)])
def test_augmented_passes_give_the_gradients(T, dk, dv, gamma, floor, phi_on):
    rng = np.random.default_rng(T * 100 + dk + 7 * floor + 3 * phi_on)
    q, k = rng.standard_normal((2, T, dk)) * 0.7
    v, dO = rng.standard_normal((2, T, dv))
    S0 = np.abs(rng.standard_normal((dk, dv))) * 0.3
    z0 = np.abs(rng.standard_normal(dk)) + 0.5
    dST = rng.standard_normal((dk, dv)) * 0.1
    dzT = rng.standard_normal(dk) * 0.1
    eps = 1e-6
    kw = dict(phi=phi_on, normalize=True, eps=eps, floor=floor)
    qt, kt = (phi(q), phi(k)) if phi_on else (q, k)
    # the forward pass's per-token denominators and du, from the oracle's outputs
    O, _, _ = oracle.recurrent(q[None, None], k[None, None], v[None, None], [gamma],
                               S0=S0[None, None], z0=z0[None, None], **kw)
    o = O[0, 0]
    z = np.zeros((T, dk))
    zz = z0.copy()
    for t in range(T):
        zz = gamma * zz + kt[t]
        z[t] = zz
    u = (qt * z).sum(1)
    if floor:
        dd = np.maximum(np.abs(u), 1.0)
        ddu = np.where(np.abs(u) > 1.0, np.sign(u), 0.0)
    else:
        dd = u + eps
        ddu = np.ones(T)
    dn = dO / dd[:, None]
    du = -(dO * o).sum(1) / dd * ddu
    du_hi = np.round(du, 3)
    du_lo = du - du_hi
    ones = np.ones((T, 1))
    Xq = np.hstack([dn, du_hi[:, None], du_lo[:, None]])
    Xk = np.hstack([v, ones, ones])
    s0 = np.vstack([S0.T, z0[None], z0[None]])
    gk0 = np.vstack([dST.T, dzT[None], np.zeros((1, dk))]) / gamma
    dqt, _ = forward(Xq, Xk, kt, gamma, s0)
    dkt, gk_fin = reversed_forward(Xk, Xq, qt, gamma, gk0)
    dv_, g_fin = reversed_forward(kt, qt, dn, gamma, dST / gamma)
    dphi_q = np.where(q > 0, 1.0, np.exp(np.minimum(q, 0.0))) if phi_on else np.ones_like(q)
    dphi_k = np.where(k > 0, 1.0, np.exp(np.minimum(k, 0.0))) if phi_on else np.ones_like(k)
    dq, dk_ = dqt * dphi_q, dkt * dphi_k
    dS0 = gamma * g_fin
    dz0 = gamma * (gk_fin[dv] + gk_fin[dv + 1])
    rq, rk, rv, rS0, rz0 = oracle.recurrent_bwd(
        q[None, None], k[None, None], v[None, None], [gamma], dO[None, None], S0=S0[None, None],
        z0=z0[None, None], dS_T=dST[None, None], dz_T=dzT[None, None], **kw)
    np.testing.assert_allclose(dq, rq[0, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk_, rk[0, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv_, rv[0, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dS0, rS0[0, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dz0, rz0[0, 0], rtol=1e-9, atol=1e-11)
