"""The segment plan's state fold, checked on the host in fp64.

A long sequence is cut into P segments of a common length (the last one may be
shorter).  The state walk computes each segment's own contribution agg_q (its state
from a zero start) and, with per-token decays, its total decay.  The entry states
are then folded:

  entry_0 = S_0,  entry_(q+1) = (decay over segment q) * entry_q + agg_q,

with the decay gamma^len for a per-head decay, or the product of the segment's
a_t.  The output walk restarts every segment from its entry state.  This is the
recurrence S_t = a_t S_(t-1) + k_t^T v_t unrolled over a segment (the chunkwise
form of the "RetNet" and "Linear attention" pages, one level up).  Here each
piece is an oracle call on a slice, and the fold must reproduce the oracle's
single pass over the whole sequence.
"""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("gated", [False, True], ids=["gamma", "gated"])
@pytest.mark.parametrize("T,seg_len", [(300, 128), (256, 64), (129, 64)])
def test_folded_entry_states_reproduce_one_pass(T, seg_len, gated):
    dk, dv, gamma = 6, 5, 0.97
    rng = np.random.default_rng(T + seg_len)
    q, k = rng.standard_normal((2, 1, 1, T, dk))
    v = rng.standard_normal((1, 1, T, dv))
    log_a = np.log(rng.uniform(0.8, 1.0, (1, 1, T))) if gated else None
    S0 = rng.standard_normal((1, 1, dk, dv)) * 0.3
    z0 = np.abs(rng.standard_normal((1, 1, dk)))

    def run(sl, S_in, z_in):
        kw = dict(normalize=True, eps=1e-6, S0=S_in, z0=z_in)
        if gated:
            return oracle.recurrent_gated(q[..., sl, :], k[..., sl, :], v[..., sl, :],
                                          log_a[..., sl], **kw)
        return oracle.recurrent(q[..., sl, :], k[..., sl, :], v[..., sl, :], [gamma], **kw)

    O_ref, S_ref, z_ref = run(slice(0, T), S0, z0)
    P = -(-T // seg_len)
    entry, zentry = S0, z0
    for qi in range(P):
        sl = slice(qi * seg_len, min(T, (qi + 1) * seg_len))
        O, S, z = run(sl, entry, zentry)  # the output walk from the entry state
        np.testing.assert_allclose(O, O_ref[..., sl, :], rtol=1e-10, atol=1e-12)
        if qi + 1 == P:
            np.testing.assert_allclose(S, S_ref, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(z, z_ref, rtol=1e-10, atol=1e-12)
            break
        _, agg, zagg = run(sl, np.zeros_like(S0), np.zeros_like(z0))  # the state walk
        decay = np.exp(log_a[..., sl].sum()) if gated else gamma ** (sl.stop - sl.start)
        entry, zentry = decay * entry + agg, decay * zentry + zagg
