"""The Taylor kernel's on-chip compression, checked on the host in fp64.

The page's map ("Linear attention" page, "A Taylor feature map") has 1 + d + d^2
features: the constant, x, and every ordered product x_a x_b / sqrt(2).  Since
x_a x_b = x_b x_a, the kernel keeps one feature per unordered pair instead:
x_a x_b for a < b and x_a^2 / sqrt(2) for a = b, 1 + d + d(d+1)/2 features in
all (153 for d = 16).  The dot products are the same, so the outputs are too.  The
state it carries is the symmetric part of the page's.  Every update k k^T is
symmetric, so the page-order final state is the symmetric part rebuilt from the
compressed state plus the initial state's antisymmetric part, decayed by
gamma^T.  These tests check both claims against the oracle, which uses the
page's features.
"""
import numpy as np
import pytest

import oracle


def compressed_features(x):
    """[n][d] -> [n][1 + d + d(d+1)/2]: 1, x, then (a, b) for a <= b, a-major."""
    n, d = x.shape
    cols = [np.ones((n, 1)), x]
    for a in range(d):
        for b in range(a, d):
            cols.append((x[:, a] * x[:, b] / (np.sqrt(2.0) if a == b else 1.0))[:, None])
    return np.concatenate(cols, axis=1)


def compress_state(S0, d):
    """A page-order state [1 + d + d^2][dv] -> the compressed rows that give the same
    read-out q~^T S for every q (pair rows: (S0[ab] + S0[ba]) / sqrt(2))."""
    rows = [S0[0], *S0[1:1 + d]]
    for a in range(d):
        for b in range(a, d):
            ra, rb = 1 + d + a * d + b, 1 + d + b * d + a
            rows.append(S0[ra] if a == b else (S0[ra] + S0[rb]) / np.sqrt(2.0))
    return np.stack(rows)


def rebuild_state(C, S0, gamma, T, d):
    """The compressed final state C and the page-order initial state S0 -> the
    page-order final state."""
    S = np.zeros_like(S0)
    S[:1 + d] = C[:1 + d]
    p = 1 + d
    for a in range(d):
        for b in range(a, d):
            ra, rb = 1 + d + a * d + b, 1 + d + b * d + a
            if a == b:
                S[ra] = C[p]
            else:
                anti = gamma ** T * (S0[ra] - S0[rb]) / 2.0
                S[ra] = C[p] / np.sqrt(2.0) + anti
                S[rb] = C[p] / np.sqrt(2.0) - anti
            p += 1
    return S


def test_compressed_features_have_the_pages_dot_products():
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((2, 50, 16)) * 0.5
    s = np.sum(q * k, axis=1)
    cq, ck = compressed_features(q), compressed_features(k)
    assert cq.shape[1] == 153
    np.testing.assert_allclose(np.sum(cq * ck, axis=1), 1 + s + s * s / 2, rtol=1e-13)


@pytest.mark.parametrize("T,gamma,normalize", [(1, 1.0, True), (40, 1.0, True), (33, 0.95, False),
                                               (64, 0.8, True)])
def test_compressed_recurrence_equals_the_page_order_oracle(T, gamma, normalize):
    d, dv = 4, 5
    rng = np.random.default_rng(T)
    q, k = rng.standard_normal((2, 1, 1, T, d)) * 0.5
    v = rng.standard_normal((1, 1, T, dv))
    df = 1 + d + d * d
    S0 = rng.standard_normal((1, 1, df, dv)) * 0.2  # not symmetric in its pair rows
    z0 = np.abs(rng.standard_normal((1, 1, df))) * 0.2
    O, S, z = oracle.recurrent_taylor(q, k, v, [gamma], normalize=normalize, eps=0.0,
                                      S0=S0, z0=z0 if normalize else None)
    cq, ck = compressed_features(q[0, 0]), compressed_features(k[0, 0])
    C0 = compress_state(S0[0, 0], d)
    c0 = compress_state(z0[0, 0][:, None], d)[:, 0]
    Oc, Cs, cz = oracle.recurrent(cq[None, None], ck[None, None], v, [gamma],
                                  normalize=normalize, eps=0.0, S0=C0[None, None],
                                  z0=c0[None, None] if normalize else None)
    np.testing.assert_allclose(Oc, O, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(rebuild_state(Cs[0, 0], S0[0, 0], gamma, T, d), S[0, 0],
                               rtol=1e-11, atol=1e-12)
    if normalize:
        zr = rebuild_state(cz[0, 0][:, None], z0[0, 0][:, None], gamma, T, d)[:, 0]
        np.testing.assert_allclose(zr, z[0, 0], rtol=1e-11, atol=1e-12)
