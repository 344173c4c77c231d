"""Independent computations that pin the oracle (test helpers, fp64 numpy).

None of these calls the oracle or the CUDA path.  Each restates a form the
pages give (or the mathematics fixes) in a different way from the oracle's
token-by-token recurrence:

* ``parallel_form``: the masked quadratic form.  "RetNet" (bembew), section
  "Parallel Representation": O = (Q K^T . D) V with D_nm = gamma^(n-m) for
  n >= m, else 0.  With phi and the normaliser it is the theorem "Recurrent and
  parallel forms agree" of the "Linear attention" page (zerotofrontier 21.2):
  O = diag(W 1)^-1 W V with W = (phi(Q) phi(K)^T) . L; for gamma < 1 the mask
  L is replaced by D (the reading that z decays with gamma).
  With ``floor`` each row of W is divided by max(|row sum|, 1) instead: RetNet's
  row normalisation of its scores ("Its normalizer is unstable" on the "Linear
  attention" page: each row divided by the absolute value of its sum, clamped
  below at 1).
* ``noncausal_left`` / ``noncausal_right``: the two multiplication orders of
  "Moving the parentheses" on the "Linear attention" page.
* ``chunkwise``: the chunkwise form that the pages describe only in words
  ("Chunked Recurrent Representation" on the "RetNet" page; "Chunkwise form"
  in section 12.5 subsection 6): parallel inside each chunk of C tokens, the
  state carried across chunks.  Written out here from the recurrence:
      O_c = ((phi(Q_c) phi(K_c)^T) . D) V_c + (phi(Q_c) . xi) S_{c-1}
      S_c = gamma^L S_{c-1} + (phi(K_c) . zeta)^T V_c
  with xi_i = gamma^(i+1), zeta_j = gamma^(L-1-j), L the chunk's length.
* ``parallel_form_gated``: the same masked quadratic form with a per-token
  decay a_t (the gate G_t = a_t 1 of "Gated Linear Attention" in section 12.5
  and of the generic loop of section 13.3 subsection 4): D[n, m] is the
  product a_{m+1} ... a_n, formed by explicit products, and the initial state
  enters as (a_0 ... a_n) q_n S_0.
* ``chunkwise_gated``: the chunkwise form with that decay, from cumulative
  log-decays b_i = log a_0 + ... + log a_i inside the chunk:
  D_ij = e^(b_i - b_j), xi_i = e^(b_i), zeta_j = e^(b_(L-1) - b_j), and the
  chunk's decay e^(b_(L-1)) in place of gamma^L.
"""
from __future__ import annotations

import numpy as np


def phi_elu1(x: np.ndarray) -> np.ndarray:
    """elu(x) + 1 written from its two branches (x + 1 above 0, e^x below)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _phi(x, phi):
    return phi_elu1(x) if phi else np.asarray(x, dtype=np.float64)


def decay_mask(T: int, gamma: float) -> np.ndarray:
    """D[n, m] = gamma^(n-m) for n >= m, 0 otherwise."""
    n = np.arange(T)[:, None]
    m = np.arange(T)[None, :]
    diff = n - m
    return np.where(diff >= 0, np.power(float(gamma), np.maximum(diff, 0)), 0.0)


def parallel_form(q, k, v, gamma, phi=False, normalize=False, eps=1e-6, floor=False):
    """Masked quadratic form for [B,H,T,d] inputs; returns O [B,H,T,dv]."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    B, H, T, _ = q.shape
    g = np.broadcast_to(np.asarray(gamma, dtype=np.float64).reshape(-1), (H,))
    out = np.empty(q.shape[:3] + (v.shape[-1],))
    for b in range(B):
        for h in range(H):
            W = (_phi(q[b, h], phi) @ _phi(k[b, h], phi).T) * decay_mask(T, g[h])
            if floor:  # each score row scaled by 1 / max(|its sum|, 1), then times V
                W = W / np.maximum(np.abs(W.sum(axis=1, keepdims=True)), 1.0)
            O = W @ v[b, h]
            if normalize and not floor:
                O = O / (W.sum(axis=1, keepdims=True) + eps)
            out[b, h] = O
    return out


def gated_mask(a) -> np.ndarray:
    """D[n, m] = a[m+1] * ... * a[n] for n >= m (1 on the diagonal), 0 above it."""
    a = np.asarray(a, dtype=np.float64)
    T = a.shape[0]
    D = np.zeros((T, T))
    for n in range(T):
        p = 1.0
        D[n, n] = 1.0
        for m in range(n - 1, -1, -1):
            p *= a[m + 1]
            D[n, m] = p
    return D


def parallel_form_gated(q, k, v, log_a, phi=False, normalize=False, eps=1e-6, floor=False,
                        S0=None, z0=None):
    """Masked quadratic form with per-token decays a = exp(log_a) ([B,H,T]) and an
    optional initial state; returns O [B,H,T,dv]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    a = np.exp(np.asarray(log_a, dtype=np.float64))
    out = np.empty((B, H, T, dv))
    for b in range(B):
        for h in range(H):
            fq, fk = _phi(q[b, h], phi), _phi(k[b, h], phi)
            W = (fq @ fk.T) * gated_mask(a[b, h])
            head = np.cumprod(a[b, h])  # a_0 ... a_n: the initial state's decay at n
            num = W @ v[b, h]
            den = W.sum(axis=1)
            if S0 is not None:
                num = num + head[:, None] * (fq @ np.asarray(S0, dtype=np.float64)[b, h])
            if z0 is not None:
                den = den + head * (fq @ np.asarray(z0, dtype=np.float64)[b, h])
            if floor:
                num = num / np.maximum(np.abs(den), 1.0)[:, None]
            elif normalize:
                num = num / (den[:, None] + eps)
            out[b, h] = num
    return out


def chunkwise_gated(q, k, v, log_a, C, phi=False, normalize=False, eps=1e-6, S0=None, z0=None):
    """Chunkwise form with per-token decays (module docstring); returns (O, S_T, z_T)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    la = np.asarray(log_a, dtype=np.float64)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    O = np.zeros((B, H, T, dv))
    S_all = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    z_all = np.zeros((B, H, dk)) if z0 is None else np.array(z0, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            S, z = S_all[b, h].copy(), z_all[b, h].copy()
            for c0 in range(0, T, C):
                L = min(C, T - c0)
                Qc = _phi(q[b, h, c0:c0 + L], phi)
                Kc = _phi(k[b, h, c0:c0 + L], phi)
                Vc = v[b, h, c0:c0 + L]
                cb = np.cumsum(la[b, h, c0:c0 + L])
                diff = cb[:, None] - cb[None, :]
                D = np.where(np.tril(np.ones((L, L))) > 0, np.exp(np.minimum(diff, 0.0)), 0.0)
                xi = np.exp(cb)[:, None]
                zeta = np.exp(cb[-1] - cb)[:, None]
                A = (Qc @ Kc.T) * D
                num = A @ Vc + (Qc * xi) @ S
                if normalize:
                    den = A.sum(axis=1) + (Qc * xi) @ z
                    num = num / (den[:, None] + eps)
                O[b, h, c0:c0 + L] = num
                S = np.exp(cb[-1]) * S + (Kc * zeta).T @ Vc
                z = np.exp(cb[-1]) * z + (Kc * zeta).sum(axis=0)
            S_all[b, h], z_all[b, h] = S, z
    return O, S_all, z_all


def noncausal_left(q, k, v, phi=False, normalize=False, eps=1e-6):
    """(phi(Q) phi(K)^T) V, the left order, per (b, h)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    A = np.einsum("bhtd,bhsd->bhts", _phi(q, phi), _phi(k, phi))
    O = A @ v
    if normalize:
        O = O / (A.sum(axis=-1, keepdims=True) + eps)
    return O


def noncausal_right(q, k, v, phi=False, normalize=False, eps=1e-6):
    """phi(Q) (phi(K)^T V), the right order, per (b, h)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    fq, fk = _phi(q, phi), _phi(k, phi)
    S = np.swapaxes(fk, -1, -2) @ v
    O = fq @ S
    if normalize:
        z = fk.sum(axis=-2)  # [B,H,dk]
        O = O / (np.einsum("bhtd,bhd->bht", fq, z)[..., None] + eps)
    return O


def chunkwise(q, k, v, gamma, C, phi=False, normalize=False, eps=1e-6, S0=None, z0=None):
    """Chunkwise form (see module docstring); returns (O, S_T, z_T)."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    g = np.broadcast_to(np.asarray(gamma, dtype=np.float64).reshape(-1), (H,))
    O = np.zeros((B, H, T, dv))
    S_all = np.zeros((B, H, dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    z_all = np.zeros((B, H, dk)) if z0 is None else np.array(z0, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            S, z = S_all[b, h].copy(), z_all[b, h].copy()
            for c0 in range(0, T, C):
                L = min(C, T - c0)
                Qc = _phi(q[b, h, c0:c0 + L], phi)
                Kc = _phi(k[b, h, c0:c0 + L], phi)
                Vc = v[b, h, c0:c0 + L]
                i = np.arange(L)
                xi = np.power(g[h], i + 1.0)[:, None]
                zeta = np.power(g[h], L - 1.0 - i)[:, None]
                A = (Qc @ Kc.T) * decay_mask(L, g[h])
                num = A @ Vc + (Qc * xi) @ S
                if normalize:
                    den = A.sum(axis=1) + (Qc * xi) @ z
                    num = num / (den[:, None] + eps)
                O[b, h, c0:c0 + L] = num
                S = g[h] ** L * S + (Kc * zeta).T @ Vc
                z = g[h] ** L * z + (Kc * zeta).sum(axis=0)
            S_all[b, h], z_all[b, h] = S, z
    return O, S_all, z_all


def rel_err(a, ref) -> float:
    """max|a - ref| / max|ref| (0 when both are all zero)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(a - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)
