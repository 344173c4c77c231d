"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: the
pages' worked examples (tests/golden/), brute-force parallel forms, closed
forms, a library IIR filter, and invariants the pages state.  The last test
rebuilds the oracle with each planted mistake and shows that some pin fails.

Which pin covers which part of the oracle:
  recurrence, phi, normaliser, update order  -> hand example (exact)
  causal mask, decay exponent, d_k != d_v    -> brute-force parallel form
  decay accuracy over long T                 -> geometric-series closed form
  decay as a linear filter                   -> scipy.signal.lfilter special case
  non-causal form                            -> left/right multiplication orders
  final state                                -> associative-memory example, orthonormal keys
  normalised outputs                         -> constant V, o_1 = v_1, convex hull
  floored normaliser                         -> RetNet's clamped row sums (parallel form);
                                                plain normaliser / unnormalised read-out
                                                where the floor is inactive / active
  chunkwise equations (the CUDA path's form) -> chunk-size invariance
  state hand-off (decode, resume)            -> split prefill / decode == one pass
  per-token decay                            -> masked form with explicit gate products,
                                                constant gate == gamma, a_t = 0 resets,
                                                chunkwise equations with cumulative logs
  Taylor feature map                         -> the page's worked pair (features and kernel),
                                                the theorem 1 + s + s^2/2 and its minimum,
                                                normalised outputs as the kernel-weighted
                                                average computed from s alone, state rows
                                                as explicit sums
"""
import json
import os

import numpy as np
import pytest

import oracle
import pins
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# pin functions: each takes an oracle library handle (None = the real one) and
# raises AssertionError on a mismatch.  The mutant test reuses them.
# ---------------------------------------------------------------------------

def pin_hand_example(lib=None):
    g = _golden("hand_example_three_tokens.json")
    q, k, v = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v"))
    O, S, z = oracle.recurrent(q, k, v, 1.0, phi=True, normalize=True, eps=0.0, _lib=lib)
    want = np.array([[a / b for a, b in row] for row in g["o_fraction"]])
    np.testing.assert_allclose(O[0, 0], want, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(S[0, 0], np.array(g["S"][-1], dtype=np.float64))
    np.testing.assert_array_equal(z[0, 0], np.array(g["z"][-1], dtype=np.float64))
    # every intermediate state, one token at a time
    for t in range(3):
        O_t, S_t, z_t = oracle.recurrent(q[: t + 1], k[: t + 1], v[: t + 1], 1.0, phi=True,
                                         normalize=True, eps=0.0, _lib=lib)
        np.testing.assert_array_equal(S_t[0, 0], np.array(g["S"][t], dtype=np.float64))
        np.testing.assert_array_equal(z_t[0, 0], np.array(g["z"][t], dtype=np.float64))
        O_raw, _, _ = oracle.recurrent(q[: t + 1], k[: t + 1], v[: t + 1], 1.0, phi=True,
                                       normalize=False, _lib=lib)
        np.testing.assert_array_equal(O_raw[0, 0, t], np.array(g["numerator"][t], dtype=float))


def pin_parallel_form(lib=None):
    rng = _rng(1)
    for trial in range(6):
        B, H = 2, 3
        T = int(rng.integers(1, 48))
        dk, dv = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        if trial == 0:
            dk, dv = 3, 7  # d_k != d_v on purpose
        phi = bool(trial % 2)
        normalize = phi and trial % 4 == 1
        q = rng.standard_normal((B, H, T, dk))
        k = rng.standard_normal((B, H, T, dk))
        v = rng.standard_normal((B, H, T, dv))
        gamma = rng.uniform(0.5, 1.0, H)
        gamma[0] = 1.0
        O, _, _ = oracle.recurrent(q, k, v, gamma, phi=phi, normalize=normalize, eps=1e-6,
                                   _lib=lib)
        ref = pins.parallel_form(q, k, v, gamma, phi=phi, normalize=normalize, eps=1e-6)
        assert pins.rel_err(O, ref) < 1e-12, (trial, pins.rel_err(O, ref))


def pin_masked_kernel_theorem(lib=None):
    """diag(W1)^-1 W V with W = (phi(Q)phi(K)^T) . L equals the recurrence (gamma = 1)."""
    rng = _rng(2)
    q = rng.standard_normal((1, 2, 40, 5))
    k = rng.standard_normal((1, 2, 40, 5))
    v = rng.standard_normal((1, 2, 40, 6))
    O, _, _ = oracle.recurrent(q, k, v, 1.0, phi=True, normalize=True, eps=0.0, _lib=lib)
    ref = pins.parallel_form(q, k, v, 1.0, phi=True, normalize=True, eps=0.0)
    assert pins.rel_err(O, ref) < 1e-12


def pin_geometric_series(lib=None):
    """d = 1, q = k = v = 1: o_n = sum_{m<=n} gamma^(n-m) = (1 - gamma^(n+1)) / (1 - gamma)."""
    T = 65536
    ones = np.ones((1, 1, T, 1))
    for g in (0.99, 0.9999):
        O, S, _ = oracle.recurrent(ones, ones, ones, g, _lib=lib)
        n = np.arange(T, dtype=np.float64)
        want = -np.expm1((n + 1.0) * np.log(g)) / (1.0 - g)
        np.testing.assert_allclose(O[0, 0, :, 0], want, rtol=1e-10)
        np.testing.assert_allclose(S[0, 0, 0, 0], want[-1], rtol=1e-10)


def pin_iir_filter(lib=None):
    """Constant q = c and k = b, d_v = 1: o = (c.b) * IIR filter 1/(1 - gamma z^-1) of v.

    The scalar-decay special case of the SSD example on the "Linear Attention,
    RWKV, and RetNet" page (section 13.3), checked against scipy's lfilter.
    """
    from scipy.signal import lfilter
    rng = _rng(3)
    T, n = 200, 4
    c, b = rng.standard_normal(n), rng.standard_normal(n)
    u = rng.standard_normal(T)
    for alpha in (0.85, 0.5, 1.0):
        q = np.tile(c, (T, 1))
        k = np.tile(b, (T, 1))
        O, _, _ = oracle.recurrent(q, k, u[:, None], alpha, _lib=lib)
        want = float(c @ b) * lfilter([1.0], [1.0, -alpha], u)
        np.testing.assert_allclose(O[0, 0, :, 0], want, rtol=1e-12, atol=1e-12)


def pin_noncausal_orders(lib=None):
    rng = _rng(4)
    q = rng.standard_normal((2, 2, 33, 6))
    k = rng.standard_normal((2, 2, 33, 6))
    v = rng.standard_normal((2, 2, 33, 9))
    for phi, normalize in ((False, False), (True, False), (True, True)):
        O, S, _ = oracle.noncausal(q, k, v, phi=phi, normalize=normalize, _lib=lib)
        left = pins.noncausal_left(q, k, v, phi=phi, normalize=normalize)
        right = pins.noncausal_right(q, k, v, phi=phi, normalize=normalize)
        assert pins.rel_err(O, left) < 1e-12
        assert pins.rel_err(O, right) < 1e-12
        # its summary is the causal final state at gamma = 1
        _, S_c, _ = oracle.recurrent(q, k, v, 1.0, phi=phi, _lib=lib)
        assert pins.rel_err(S, S_c) < 1e-12


def pin_associative_memory(lib=None):
    g = _golden("associative_memory_three_pairs.json")
    k = np.array(g["k"], dtype=np.float64)
    v = np.array(g["v"], dtype=np.float64)
    O, S, _ = oracle.noncausal(k[:2], k[:2], v[:2], _lib=lib)
    np.testing.assert_allclose(S[0, 0], g["S_after_two"], atol=1e-15)
    np.testing.assert_allclose(O[0, 0, 0], g["reads_after_two"]["k1"], atol=1e-15)
    np.testing.assert_allclose(O[0, 0, 1], g["reads_after_two"]["k2"], atol=1e-15)
    O, S, _ = oracle.noncausal(k, k, v, _lib=lib)
    np.testing.assert_allclose(S[0, 0], g["S_after_three"], atol=1e-14)
    np.testing.assert_allclose(O[0, 0, 0], g["reads_after_three"]["k1"], atol=1e-14)
    np.testing.assert_allclose(O[0, 0, 2], g["reads_after_three"]["k3"], atol=1e-14)
    # the causal form reaches the same final state
    _, S_c, _ = oracle.recurrent(k, k, v, 1.0, _lib=lib)
    np.testing.assert_allclose(S_c[0, 0], g["S_after_three"], atol=1e-14)


def pin_orthonormal_keys(lib=None):
    """Orthonormal keys, gamma = 1, identity phi: each causal read returns its own value."""
    rng = _rng(5)
    dk, dv = 16, 24
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm.T  # rows orthonormal
    v = rng.standard_normal((dk, dv))
    O, S, _ = oracle.recurrent(keys, keys, v, 1.0, _lib=lib)
    np.testing.assert_allclose(O[0, 0], v, atol=1e-12)
    np.testing.assert_allclose(S[0, 0], keys.T @ v, atol=1e-12)


def pin_normalised_invariants(lib=None):
    rng = _rng(6)
    B, H, T, dk, dv = 1, 3, 64, 8, 5
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    gamma = np.array([1.0, 0.9, 0.5])
    # constant values give constant outputs (also with decay: z decays like S)
    c = rng.standard_normal(dv)
    vc = np.broadcast_to(c, (B, H, T, dv)).copy()
    O, _, _ = oracle.recurrent(q, k, vc, gamma, phi=True, normalize=True, eps=0.0, _lib=lib)
    np.testing.assert_allclose(O, vc, rtol=1e-13, atol=1e-13)
    # the first output is the first value; every output lies in the values' hull
    v = rng.standard_normal((B, H, T, dv))
    O, _, _ = oracle.recurrent(q, k, v, gamma, phi=True, normalize=True, eps=0.0, _lib=lib)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], rtol=1e-13, atol=1e-13)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(O >= lo - 1e-12) and np.all(O <= hi + 1e-12)


def pin_chunkwise_invariance(lib=None):
    rng = _rng(7)
    B, H, T, dk, dv = 2, 2, 77, 6, 10
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    gamma = np.array([0.95, 0.6])
    for phi, normalize in ((False, False), (True, True)):
        O, S, z = oracle.recurrent(q, k, v, gamma, phi=phi, normalize=normalize, _lib=lib)
        for C in (1, 4, 16, 32, 64, 128):
            Oc, Sc, zc = pins.chunkwise(q, k, v, gamma, C, phi=phi, normalize=normalize)
            assert pins.rel_err(Oc, O) < 1e-12, (C, pins.rel_err(Oc, O))
            assert pins.rel_err(Sc, S) < 1e-12
            if normalize:
                assert pins.rel_err(zc, z) < 1e-12


def pin_state_handoff(lib=None):
    """Prefill T1 then resume (chunked or token by token) equals one pass over T."""
    rng = _rng(8)
    B, H, T, dk, dv = 2, 2, 50, 4, 6
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    gamma = np.array([0.9, 1.0])
    O, S, z = oracle.recurrent(q, k, v, gamma, phi=True, normalize=True, _lib=lib)
    t1 = 31
    O1, S1, z1 = oracle.recurrent(q[:, :, :t1], k[:, :, :t1], v[:, :, :t1], gamma, phi=True,
                                  normalize=True, _lib=lib)
    O2, S2, z2 = oracle.recurrent(q[:, :, t1:], k[:, :, t1:], v[:, :, t1:], gamma, phi=True,
                                  normalize=True, S0=S1, z0=z1, _lib=lib)
    assert pins.rel_err(np.concatenate([O1, O2], axis=2), O) < 1e-13
    assert pins.rel_err(S2, S) < 1e-13 and pins.rel_err(z2, z) < 1e-13


def pin_floor_clamped_rows(lib=None):
    """Floored normaliser = RetNet's parallel form with each score row divided by
    max(|row sum|, 1); identity features of both signs, so rows with sums below
    -1, between -1 and 1, and above 1 all occur."""
    rng = _rng(31)
    B, H, T, dk, dv = 2, 3, 24, 6, 5
    q = rng.standard_normal((B, H, T, dk)) * 0.8
    k = rng.standard_normal((B, H, T, dk)) * 0.8
    v = rng.standard_normal((B, H, T, dv))
    gamma = np.array([0.9, 0.99, 1.0])
    O, _, _ = oracle.recurrent(q, k, v, gamma, floor=True, _lib=lib)
    ref = pins.parallel_form(q, k, v, gamma, floor=True)
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)
    sums = np.concatenate([((q[b, h] @ k[b, h].T) * pins.decay_mask(T, gamma[h])).sum(axis=1)
                           for b in range(B) for h in range(H)])
    assert (sums < -1).any() and (np.abs(sums) < 1).any() and (sums > 1).any()
    # the non-causal form, floored, against the left multiplication order
    On, _, _ = oracle.noncausal(q, k, v, floor=True, _lib=lib)
    A = np.einsum("bhtd,bhsd->bhts", q, k)
    A = A / np.maximum(np.abs(A.sum(axis=-1, keepdims=True)), 1.0)
    np.testing.assert_allclose(On, A @ v, rtol=1e-10, atol=1e-12)


def pin_floor_limits(lib=None):
    """Where every |q~^T z| >= 1 the floor changes nothing (the plain normaliser at
    eps = 0); where every |q~^T z| < 1 it leaves the read-out undivided."""
    rng = _rng(32)
    B, H, T, dk, dv = 1, 2, 20, 4, 3
    v = rng.standard_normal((B, H, T, dv))
    q = np.abs(rng.standard_normal((B, H, T, dk))) + 1.0   # elu+1 features >= 2
    k = np.abs(rng.standard_normal((B, H, T, dk))) + 1.0
    Of, Sf, zf = oracle.recurrent(q, k, v, 0.95, phi=True, floor=True, _lib=lib)
    On, Sn, zn = oracle.recurrent(q, k, v, 0.95, phi=True, normalize=True, eps=0.0, _lib=lib)
    np.testing.assert_allclose(Of, On, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(Sf, Sn)
    qs = rng.standard_normal((B, H, T, dk)) * 0.05          # tiny scores: |q^T z| < 1
    ks = rng.standard_normal((B, H, T, dk)) * 0.05
    Of, _, _ = oracle.recurrent(qs, ks, v, 0.95, floor=True, _lib=lib)
    Ou, _, _ = oracle.recurrent(qs, ks, v, 0.95, _lib=lib)
    np.testing.assert_allclose(Of, Ou, rtol=1e-13, atol=0)


def _gated_case(seed, B, H, T, dk, dv):
    rng = _rng(seed)
    q = rng.standard_normal((B, H, T, dk)) * 0.7
    k = rng.standard_normal((B, H, T, dk)) * 0.7
    v = rng.standard_normal((B, H, T, dv))
    log_a = -rng.exponential(0.3, (B, H, T))   # a_t in (0, 1], about 0.74 on average
    S0 = rng.standard_normal((B, H, dk, dv))
    z0 = np.abs(rng.standard_normal((B, H, dk)))
    return q, k, v, log_a, S0, z0


def pin_gated_parallel_form(lib=None):
    """Per-token decay = the masked form with D[n, m] = a_{m+1} ... a_n and the
    initial state decayed by a_0 ... a_n (explicit products), for plain, phi +
    normaliser and floored read-outs, d_k != d_v."""
    q, k, v, log_a, S0, z0 = _gated_case(41, 2, 3, 19, 5, 4)
    for phi, norm, floor in ((False, False, False), (True, True, False), (False, False, True)):
        O, _, _ = oracle.recurrent_gated(q, k, v, log_a, phi=phi, normalize=norm, floor=floor,
                                         S0=S0, z0=z0, _lib=lib)
        ref = pins.parallel_form_gated(q, k, v, log_a, phi=phi, normalize=norm, floor=floor,
                                       S0=S0, z0=z0)
        np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


def pin_gated_constant_is_gamma(lib=None):
    """A per-token decay that is the same for every token of a head is gamma."""
    q, k, v, _, S0, z0 = _gated_case(42, 2, 3, 40, 6, 6)
    gamma = np.array([0.9, 0.99, 1.0])
    log_a = np.broadcast_to(np.log(gamma)[None, :, None], (2, 3, 40))
    Og, Sg, zg = oracle.recurrent_gated(q, k, v, log_a, phi=True, normalize=True, S0=S0, z0=z0,
                                        _lib=lib)
    O, S, z = oracle.recurrent(q, k, v, gamma, phi=True, normalize=True, S0=S0, z0=z0, _lib=lib)
    for got, want in ((Og, O), (Sg, S), (zg, z)):
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def pin_gated_reset(lib=None):
    """a_t = 0 (log a_t = -1000) forgets everything before t: the rest of the
    sequence equals a fresh start at t from the zero state."""
    q, k, v, log_a, S0, z0 = _gated_case(43, 1, 2, 30, 4, 3)
    t0 = 13
    log_a = log_a.copy()
    log_a[:, :, t0] = -1000.0
    O, S, z = oracle.recurrent_gated(q, k, v, log_a, phi=True, normalize=True, S0=S0, z0=z0,
                                     _lib=lib)
    tail = log_a[:, :, t0:].copy()
    tail[:, :, 0] = 0.0
    Ot, St, zt = oracle.recurrent_gated(q[:, :, t0:], k[:, :, t0:], v[:, :, t0:], tail,
                                        phi=True, normalize=True, _lib=lib)
    np.testing.assert_allclose(O[:, :, t0:], Ot, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, St, rtol=1e-12, atol=1e-14)


def pin_gated_chunkwise(lib=None):
    """The chunkwise equations with cumulative log-decays equal the recurrence
    at every chunk length, ragged tails included."""
    q, k, v, log_a, S0, z0 = _gated_case(44, 1, 2, 45, 5, 3)
    O, S, z = oracle.recurrent_gated(q, k, v, log_a, phi=True, normalize=True, S0=S0, z0=z0,
                                     _lib=lib)
    for C in (1, 4, 16, 45, 64):
        Oc, Sc, zc = pins.chunkwise_gated(q, k, v, log_a, C, phi=True, normalize=True, S0=S0,
                                          z0=z0)
        assert pins.rel_err(Oc, O) < 1e-12 and pins.rel_err(Sc, S) < 1e-12
        assert pins.rel_err(zc, z) < 1e-12


def _loss_and_grads(q, k, v, gamma, W, WS, Wz, phi, normalize, floor, S0, z0, log_a, lib):
    """L = sum(W * O) + <WS, S_T> + <Wz, z_T> by the forward oracle, and its gradients
    by the backward oracle (dO = W, dS_T = WS, dz_T = Wz)."""
    def loss(q_, k_, v_, S0_, z0_):
        if log_a is None:
            O, S, z = oracle.recurrent(q_, k_, v_, gamma, phi=phi, normalize=normalize,
                                       floor=floor, S0=S0_, z0=z0_, _lib=lib)
        else:
            O, S, z = oracle.recurrent_gated(q_, k_, v_, log_a, phi=phi, normalize=normalize,
                                             floor=floor, S0=S0_, z0=z0_, _lib=lib)
        return float((W * O).sum() + (WS * S).sum() + (Wz * z).sum())
    grads = oracle.recurrent_bwd(q, k, v, gamma, W, phi=phi, normalize=normalize, floor=floor,
                                 S0=S0, z0=z0, dS_T=WS, dz_T=Wz, _lib=lib, log_a=log_a)
    return loss, grads


def _check_by_differences(loss, args, grads, h=1e-6, rtol=2e-6):
    """Central differences of the loss in every element of every argument."""
    for a, g in zip(args, grads):
        num = np.zeros_like(a)
        it = np.nditer(a, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = a[idx]
            a[idx] = old + h
            lp = loss(*args)
            a[idx] = old - h
            lm = loss(*args)
            a[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(num)), 1e-30)
        assert err < rtol, f"gradient differs from the central differences: {err:.2e}"


def pin_backward_by_differences(lib=None):
    """The backward sweeps against central differences of the forward oracle, for
    plain, phi + normaliser and floored read-outs, an initial state and a final-state
    gradient, and a per-token decay."""
    rng = _rng(51)
    B, H, T, dk, dv = 1, 2, 7, 3, 4
    for phi, norm, floor, gated in ((False, False, False, False), (True, True, False, False),
                                    (False, False, True, False), (True, True, False, True)):
        q = rng.standard_normal((B, H, T, dk)) * (0.6 if floor else 0.8)
        k = rng.standard_normal((B, H, T, dk)) * (0.6 if floor else 0.8)
        v = rng.standard_normal((B, H, T, dv))
        S0 = rng.standard_normal((B, H, dk, dv)) * 0.5
        z0 = np.abs(rng.standard_normal((B, H, dk))) * (0.3 if floor else 1.0) + (0.0 if floor else 0.5)
        W = rng.standard_normal((B, H, T, dv))
        WS = rng.standard_normal((B, H, dk, dv))
        Wz = rng.standard_normal((B, H, dk))
        gamma = np.array([0.9, 0.97])
        log_a = -rng.exponential(0.2, (B, H, T)) if gated else None
        loss, (dq, dk_, dv_, dS0, dz0) = _loss_and_grads(q, k, v, gamma, W, WS, Wz, phi, norm,
                                                         floor, S0, z0, log_a, lib)
        if floor:  # the differences must not straddle the floor's kink |q~^T z| = 1
            us = []
            for h in range(H):
                zz = z0[0, h].copy()
                for t in range(T):
                    zz = gamma[h] * zz + k[0, h, t]
                    us.append(abs(q[0, h, t] @ zz))
            us = np.array(us)
            assert np.all(np.abs(us - 1.0) > 1e-3)
            assert (us < 1).any() and (us > 1).any()  # both sides of the floor
        _check_by_differences(loss, [q, k, v, S0, z0], [dq, dk_, dv_, dS0, dz0])


def pin_taylor_pair(lib=None):
    """The page's worked pair q = (1, 2), k = (3, 1): the features in the box's order
    (constant, linear, the outer product row-major over sqrt 2) and the kernel value."""
    g = _golden("taylor_features_pair.json")
    f = oracle.taylor_features(np.array([g["q"], g["k"]], float), _lib=lib)
    r2 = np.sqrt(2.0)
    np.testing.assert_allclose(f[0], [1.0, *g["q"], *(np.array(g["vec_qq"]) / r2)], rtol=1e-15)
    np.testing.assert_allclose(f[1], [1.0, *g["k"], *(np.array(g["vec_kk"]) / r2)], rtol=1e-15)
    assert abs(f[0] @ f[1] - g["kernel"]) < 1e-12
    assert g["kernel"] == 1 + g["s"] + g["s_squared"] / 2 and g["vec_dot"] == g["s_squared"]


def pin_taylor_kernel_theorem(lib=None):
    """phi(q)^T phi(k) = 1 + s + s^2/2 = ((s + 1)^2 + 1)/2 for random pairs (the page's
    theorem), and the minimum 1/2 at s = -1."""
    rng = _rng(61)
    for d in (1, 3, 16):
        q, k = rng.standard_normal((2, 50, d))
        s = np.einsum("nd,nd->n", q, k)
        fq, fk = oracle.taylor_features(q, _lib=lib), oracle.taylor_features(k, _lib=lib)
        assert fq.shape == (50, 1 + d + d * d)
        np.testing.assert_allclose(np.einsum("nf,nf->n", fq, fk), 1 + s + s * s / 2, rtol=1e-12)
    x = np.array([[1.0, 0.0]])
    fm = oracle.taylor_features(-x, _lib=lib)[0] @ oracle.taylor_features(x, _lib=lib)[0]
    assert abs(fm - 0.5) < 1e-15


def pin_taylor_attention(lib=None):
    """Causal normalised attention with the Taylor features and a per-head decay equals
    the kernel-weighted average sum_s g^(t-s) kappa(q_t, k_s) v_s / sum_s g^(t-s)
    kappa(q_t, k_s), kappa = 1 + s + s^2/2 taken from the dot products alone; the final
    state's rows are the explicit decayed sums of 1, k_i and k_i k_j / sqrt 2 times v."""
    rng = _rng(62)
    B, H, T, d, dv = 1, 2, 23, 4, 3
    q, k = rng.standard_normal((2, B, H, T, d)) * 0.7
    v = rng.standard_normal((B, H, T, dv))
    gamma = np.array([1.0, 0.9])
    O, S, z = oracle.recurrent_taylor(q, k, v, gamma, normalize=True, eps=0.0, _lib=lib)
    for h in range(H):
        sc = q[0, h] @ k[0, h].T
        kap = 1 + sc + sc * sc / 2
        n = np.arange(T)
        D = np.where(n[:, None] >= n[None, :], gamma[h] ** (n[:, None] - n[None, :]), 0.0)
        W = kap * D
        np.testing.assert_allclose(O[0, h], (W @ v[0, h]) / W.sum(1, keepdims=True), rtol=1e-11)
        w = gamma[h] ** (T - 1 - n)
        kk = k[0, h]
        np.testing.assert_allclose(S[0, h, 0], w @ v[0, h], rtol=1e-11)
        np.testing.assert_allclose(S[0, h, 1:1 + d], (kk * w[:, None]).T @ v[0, h], rtol=1e-11)
        quad = np.einsum("t,ti,tj,tv->ijv", w, kk, kk, v[0, h]) / np.sqrt(2.0)
        np.testing.assert_allclose(S[0, h, 1 + d:].reshape(d, d, dv), quad, rtol=1e-11)
        np.testing.assert_allclose(z[0, h, 0], w.sum(), rtol=1e-12)


def pin_taylor_backward_by_differences(lib=None):
    """The Taylor map's gradients (q, k through the feature map, v, the initial state
    of the features' rows) against central differences of the forward oracle with
    the map, normalised and with a per-head decay."""
    rng = _rng(63)
    B, H, T, d, dv = 1, 2, 6, 2, 3
    df = 1 + d + d * d
    q = rng.standard_normal((B, H, T, d)) * 0.7
    k = rng.standard_normal((B, H, T, d)) * 0.7
    v = rng.standard_normal((B, H, T, dv))
    S0 = rng.standard_normal((B, H, df, dv)) * 0.3
    z0 = np.abs(rng.standard_normal((B, H, df))) + 0.5
    W = rng.standard_normal((B, H, T, dv))
    WS = rng.standard_normal((B, H, df, dv))
    Wz = rng.standard_normal((B, H, df))
    gamma = np.array([1.0, 0.93])

    def loss(q_, k_, v_, S0_, z0_):
        O, S, z = oracle.recurrent_taylor(q_, k_, v_, gamma, normalize=True, S0=S0_, z0=z0_,
                                          _lib=lib)
        return float((W * O).sum() + (WS * S).sum() + (Wz * z).sum())
    grads = oracle.recurrent_bwd_taylor(q, k, v, gamma, W, normalize=True, S0=S0, z0=z0,
                                        dS_T=WS, dz_T=Wz, _lib=lib)
    _check_by_differences(loss, [q, k, v, S0, z0], grads)


ALL_PINS = [pin_hand_example, pin_parallel_form, pin_masked_kernel_theorem,
            pin_geometric_series, pin_iir_filter, pin_noncausal_orders,
            pin_associative_memory, pin_orthonormal_keys, pin_normalised_invariants,
            pin_chunkwise_invariance, pin_state_handoff, pin_floor_clamped_rows,
            pin_floor_limits, pin_gated_parallel_form, pin_gated_constant_is_gamma,
            pin_gated_reset, pin_gated_chunkwise, pin_backward_by_differences,
            pin_taylor_pair, pin_taylor_kernel_theorem, pin_taylor_attention,
            pin_taylor_backward_by_differences]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_decode_step_matches_recurrence():
    rng = _rng(9)
    B, H, T, dk, dv = 2, 3, 12, 5, 7
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    gamma = np.array([0.9, 0.99, 1.0])
    O, S, z = oracle.recurrent(q, k, v, gamma, phi=True, normalize=True)
    S_t = np.zeros((B, H, dk, dv))
    z_t = np.zeros((B, H, dk))
    for t in range(T):
        S_in = S_t.copy()
        o, S_t, z_t = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], gamma, S_t, z_t,
                                         phi=True, normalize=True)
        np.testing.assert_array_equal(S_in, S_in)  # inputs untouched
        assert pins.rel_err(o, O[:, :, t]) < 1e-13
    assert pins.rel_err(S_t, S) < 1e-13


def test_hand_example_kernel_matrix_pins_the_helper():
    """The brute-force helper reproduces the page's kernel matrix and row sums."""
    g = _golden("hand_example_three_tokens.json")
    fq = pins.phi_elu1(np.array(g["q"], dtype=float))
    fk = pins.phi_elu1(np.array(g["k"], dtype=float))
    np.testing.assert_array_equal(fq, g["phi_q"])
    np.testing.assert_array_equal(fk, g["phi_k"])
    W = fq @ fk.T
    np.testing.assert_array_equal(W, g["kernel_matrix"])
    np.testing.assert_array_equal((W * pins.decay_mask(3, 1.0)).sum(axis=1),
                                  g["masked_row_sums"])


def test_empty_sequence_returns_initial_state():
    S0 = np.arange(12, dtype=float).reshape(1, 1, 3, 4)
    z0 = np.arange(3, dtype=float).reshape(1, 1, 3)
    e = np.zeros((1, 1, 0, 3))
    O, S, z = oracle.recurrent(e, e, np.zeros((1, 1, 0, 4)), 0.9, S0=S0, z0=z0)
    assert O.shape == (1, 1, 0, 4)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_array_equal(z, z0)


def test_workload_decays_are_exact():
    """gamma_h = 1 - 2^(-5-h) ("RetNet" page, "Multi-Scale Retention") is exact in fp32."""
    g = workloads.gammas(workloads.CONFIGS["msr_retention_bf16"])
    for h, x in enumerate(g):
        assert float(x) == 1.0 - 2.0 ** (-5 - h)
    g = workloads.gammas(workloads.CONFIGS["decode_bf16"])
    assert [float(x) for x in g] == [1.0 - 2.0 ** (-5 - (h % 8)) for h in range(32)]
    g = workloads.gammas(workloads.CONFIGS["long_retention_bf16"])
    assert np.all((g >= np.float32(0.99)) & (g <= np.float32(0.9999)))


def test_input_slices_regenerate_exactly():
    full = workloads.make_inputs("linear_attention_bf16")
    pairs = [(0, 0), (2, 5), (3, 7)]
    part = workloads.make_inputs("linear_attention_bf16", pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        for n in ("q", "k", "v"):
            assert (part[n][i] == full[n][b, h]).all()


MUTANTS = {
    1: "read before write",
    2: "decay applied to the new term",
    3: "decay dropped",
    4: "normaliser not decayed",
    5: "outer product transposed",
    6: "elu without +1",
    7: "normaliser over the wrong axis",
    8: "floor without the absolute value",
    9: "per-token gate one token late",
    10: "backward sweep without the decay",
    11: "dq without the normaliser's term",
    12: "Taylor features without the 1/sqrt(2)",
    13: "eps left out of the denominator",
    14: "non-causal summary without the last token",
    15: "backward reads G before the token's own term",
    16: "dk without the chain rule through phi",
    17: "Taylor features without the constant",
    18: "Taylor features without the linear part",
    19: "Taylor map's gradient with one half of the outer product",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_planted_mistake_is_caught(mutant, tmp_path):
    lib = oracle.load_mutant(mutant, str(tmp_path))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
