"""The backward pass's segment plan, checked on the host in fp64.

The backward pass's two sweeps carry a state chunk by chunk: forward in time the
state S (for the queries' gradients), backward in time its gradient G = dL/dS
(for the keys' and values' gradients).  With a sequence cut into P segments, each
sweep restarts every segment from an entry state folded from the segments'
own contributions:

  forward:  S_entry(0) = S_0,  S_entry(q+1) = d(q) S_entry(q) + agg(q)
  backward: G_end(P-1) = dS_T, G_end(q) = d(q+1) G_end(q+1) + gagg(q+1)

with d(q) the state's decay over segment q (gamma^len, or the product of the
segment's a_t), agg(q) segment q's state from a zero start, and gagg(q) the
gradient of the loss terms of segment q's outputs with respect to the state
entering it (the same holds for z and its gradient).  This is the chain rule
through S_end(q+1) = d(q+1) S_end(q) + (terms free of S_end(q)) ("Linear
attention" page, "Decoding, training, and what each costs": the gradients are
cumulative sums running backward in time).  Here each piece is an oracle call on
a slice; the segment-wise gradients must reproduce the oracle's single pass.
"""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("normalize", [False, True], ids=["plain", "normalised"])
@pytest.mark.parametrize("gated", [False, True], ids=["gamma", "gated"])
@pytest.mark.parametrize("T,seg_len", [(300, 128), (256, 64), (129, 64)])
def test_segmented_backward_reproduces_one_pass(T, seg_len, gated, normalize):
    dk, dv, gamma = 5, 4, 0.97
    rng = np.random.default_rng(T * 7 + seg_len + gated + 2 * normalize)
    q, k = rng.standard_normal((2, 1, 1, T, dk)) * 0.5
    v = rng.standard_normal((1, 1, T, dv))
    dO = rng.standard_normal((1, 1, T, dv))
    log_a = np.log(rng.uniform(0.8, 1.0, (1, 1, T))) if gated else None
    S0 = rng.standard_normal((1, 1, dk, dv)) * 0.3
    z0 = np.abs(rng.standard_normal((1, 1, dk))) + 0.5
    dST = rng.standard_normal((1, 1, dk, dv)) * 0.2
    dzT = rng.standard_normal((1, 1, dk)) * 0.2 if normalize else None
    kw = dict(phi=normalize, normalize=normalize, eps=1e-6)

    def fwd(sl, S_in, z_in):
        if gated:
            return oracle.recurrent_gated(q[..., sl, :], k[..., sl, :], v[..., sl, :],
                                          log_a[..., sl], S0=S_in, z0=z_in, **kw)
        return oracle.recurrent(q[..., sl, :], k[..., sl, :], v[..., sl, :], [gamma], S0=S_in,
                                z0=z_in, **kw)

    def bwd(sl, S_in, z_in, G, Gz):
        return oracle.recurrent_bwd(q[..., sl, :], k[..., sl, :], v[..., sl, :], [gamma],
                                    dO[..., sl, :], S0=S_in, z0=z_in, dS_T=G, dz_T=Gz,
                                    log_a=None if log_a is None else log_a[..., sl], **kw)

    ref = bwd(slice(0, T), S0, z0, dST, dzT)
    P = -(-T // seg_len)
    sls = [slice(i * seg_len, min(T, (i + 1) * seg_len)) for i in range(P)]
    dec = [np.exp(log_a[..., s].sum()) if gated else gamma ** (s.stop - s.start) for s in sls]
    # forward fold: entry states from the segments' own contributions
    entry, zentry = [S0], [z0]
    for i in range(P - 1):
        _, agg, zagg = fwd(sls[i], np.zeros_like(S0), np.zeros_like(z0))
        entry.append(dec[i] * entry[-1] + agg)
        zentry.append(dec[i] * zentry[-1] + zagg)
    # backward fold: the state's gradient at each segment's end
    zero_g = np.zeros_like(dST)
    zero_gz = None if dzT is None else np.zeros_like(dzT)
    G_end, Gz_end = [None] * P, [None] * P
    G_end[P - 1] = dST
    Gz_end[P - 1] = np.zeros_like(z0) if dzT is None else dzT
    for i in range(P - 2, -1, -1):
        _, _, _, gagg, gzagg = bwd(sls[i + 1], entry[i + 1], zentry[i + 1], zero_g, zero_gz)
        G_end[i] = dec[i + 1] * G_end[i + 1] + gagg
        Gz_end[i] = dec[i + 1] * Gz_end[i + 1] + gzagg
    for i, s in enumerate(sls):
        dq, dk_, dv_, dS0, dz0 = bwd(s, entry[i], zentry[i], G_end[i], Gz_end[i])
        np.testing.assert_allclose(dq, ref[0][..., s, :], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(dk_, ref[1][..., s, :], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(dv_, ref[2][..., s, :], rtol=1e-9, atol=1e-11)
        if i == 0:
            np.testing.assert_allclose(dS0, ref[3], rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dz0, ref[4], rtol=1e-9, atol=1e-11)
