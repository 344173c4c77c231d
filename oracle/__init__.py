"""TEST INFRASTRUCTURE ONLY - fp64 CPU oracle for causal decayed linear attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import this
package.  The product package ``retnet_retention_gb300`` never imports it and
shares no code with it.

The arithmetic lives in ``linattn_oracle.c`` (plain C, fp64, OpenMP over the
independent (b, h) sequences); this module only marshals numpy arrays.
Every input is widened to fp64 from the exact values handed to the GPU
(bf16 or fp32), and gamma is the same fp32 number, widened.

Functions
---------
recurrent(q, k, v, gamma, phi, normalize, eps, S0, z0)
    The causal recurrent form: S = gamma S + phi(k) v^T, z = gamma z + phi(k),
    o = phi(q)^T S [/ (phi(q)^T z + eps)], update before read.  Sources:
    "Linear attention" (zerotofrontier 21.2) box "Causal linear attention,
    recurrent form"; "RetNet" (bembew) section "Recurrent Representation".
recurrent_gated(q, k, v, log_a, phi, normalize, eps, S0, z0)
    The same recurrence with a per-token decay a_t = exp(log_a[b, h, t]) in
    place of gamma: the generic "decay the old state, add, read out" loop of
    "Linear Attention, RWKV, and RetNet" (temporalbook 13.3, subsection 4)
    with the gate G_t = a_t 1 that depends on the token ("Efficient and Sparse
    Transformers", temporalbook 12.5, "Gated Linear Attention").
recurrent_bwd(q, k, v, gamma, dO, ..., log_a, dS_T, dz_T)
    Gradients of ``recurrent`` (dq, dk, dv and those of the initial state) for
    the loss sum(dO * O) + <dS_T, S_T> + <dz_T, z_T>, as two sweeps of
    cumulative sums, forward in time for the queries and backward for the keys
    and values ("Linear attention" page, "Decoding, training, and what each
    costs"); no state is stored.
decode_step(q, k, v, gamma, S, z, phi, normalize, eps)
    One token of the same recurrence: the interview box "Causal linear
    attention, recurrent and parallel, plus the decode step" on the "Linear
    attention" page.  It is ``recurrent`` with T = 1 and the state passed in.
taylor_features(x), recurrent_taylor(q, k, v, gamma, normalize, ...)
    The second-order Taylor feature map phi(x) = (1, x, vec(x x^T)/sqrt(2)) of
    the "Linear attention" page (box "Taylor features"), and ``recurrent`` on
    the features it gives (d_phi = 1 + d + d^2; d = 16 gives 273).
taylor_features_bwd(x, dfeat), recurrent_bwd_taylor(q, k, v, gamma, dO, ...)
    The map's transpose Jacobian, and the gradients of ``recurrent_taylor``:
    ``recurrent_bwd`` on the features, then the chain rule through the map.
noncausal(q, k, v, phi, normalize, eps)
    gamma = 1, every query reads the one summary phi(K)^T V: box "Linear
    attention" on the "Linear attention" page.

Each takes ``floor=True`` for the floored normaliser, o / max(|phi(q)^T z|, 1):
the matrix LSTM of the box "An LSTM whose cell is linear attention" on the
"Linear attention" page, which equals RetNet's division of each score row by
the absolute value of its sum, clamped below at 1 (same page, "Its normalizer
is unstable").

Pins: every function here is checked in ``tests/test_oracle.py`` against the
pages' worked example, brute-force parallel forms, closed forms, a library
IIR filter and invariants; see that file for which pin covers which part.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

_LIB = None


def _load(path: str | None = None):
    lib = ctypes.CDLL(path or _build.build())
    dp = ctypes.POINTER(ctypes.c_double)
    L = ctypes.c_long
    lib.oracle_recurrent.argtypes = [dp, dp, dp, dp, L, L, L, L, L, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, dp]
    lib.oracle_recurrent.restype = ctypes.c_int
    lib.oracle_recurrent_gated.argtypes = lib.oracle_recurrent.argtypes
    lib.oracle_recurrent_gated.restype = ctypes.c_int
    lib.oracle_recurrent_bwd.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, dp,
                                         dp, dp, dp, dp, dp]
    lib.oracle_recurrent_bwd.restype = ctypes.c_int
    lib.oracle_noncausal.argtypes = [dp, dp, dp, L, L, L, L, L, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, dp, dp, dp]
    lib.oracle_noncausal.restype = ctypes.c_int
    lib.oracle_taylor_features.argtypes = [dp, L, L, dp]
    lib.oracle_taylor_features.restype = None
    lib.oracle_taylor_features_bwd.argtypes = [dp, dp, L, L, dp]
    lib.oracle_taylor_features_bwd.restype = None
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def lib():
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def num_threads() -> int:
    """Threads the oracle's OpenMP loop uses on this host."""
    return int(lib().oracle_num_threads())


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: widen its exact values
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as4(x: np.ndarray, name: str) -> np.ndarray:
    if x.ndim == 2:
        x = x[None, None]
    elif x.ndim == 3:
        x = x[None]
    if x.ndim != 4:
        raise ValueError(f"{name}: expected [B,H,T,d] (or [T,d] / [H,T,d]), got {x.shape}")
    return np.ascontiguousarray(x)


def _norm_mode(normalize: bool, floor: bool) -> int:
    return 2 if floor else (1 if normalize else 0)


def recurrent(q, k, v, gamma, phi: bool = False, normalize: bool = False,
              eps: float = 1e-6, S0=None, z0=None, _lib=None, floor: bool = False):
    """Causal recurrent form in fp64.

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; gamma: [H] (or a scalar).
    S0: [B,H,dk,dv] or None; z0: [B,H,dk] or None.
    floor: divide by max(|q~^T z|, 1) instead (implies normalising; no eps).
    Returns (O [B,H,T,dv], S_T [B,H,dk,dv], z_T [B,H,dk]) as float64 arrays.
    """
    Q, K, V = _as4(_f64(q), "q"), _as4(_f64(k), "k"), _as4(_f64(v), "v")
    B, H, T, dk = Q.shape
    dv = V.shape[-1]
    if K.shape != Q.shape or V.shape[:3] != Q.shape[:3]:
        raise ValueError(f"shape mismatch q{Q.shape} k{K.shape} v{V.shape}")
    g = np.ascontiguousarray(np.broadcast_to(_f64(gamma).reshape(-1), (H,)).astype(np.float64))
    S0a = None if S0 is None else np.ascontiguousarray(_f64(S0).reshape(B, H, dk, dv))
    z0a = None if z0 is None else np.ascontiguousarray(_f64(z0).reshape(B, H, dk))
    O = np.empty((B, H, T, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    rc = (_lib or lib()).oracle_recurrent(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(g), B, H, T, dk, dv, int(bool(phi)),
        _norm_mode(normalize, floor), float(eps), _ptr(S0a), _ptr(z0a), _ptr(O), _ptr(S), _ptr(z))
    if rc != 0:
        raise MemoryError("oracle_recurrent: scratch allocation failed")
    return O, S, z


def recurrent_gated(q, k, v, log_a, phi: bool = False, normalize: bool = False,
                    eps: float = 1e-6, S0=None, z0=None, _lib=None, floor: bool = False):
    """Causal recurrent form with a per-token decay, in fp64.

    log_a: [B,H,T] natural log of a_t (the decay applied to the state before
    token t is added); the other arguments and the results as ``recurrent``.
    """
    Q, K, V = _as4(_f64(q), "q"), _as4(_f64(k), "k"), _as4(_f64(v), "v")
    B, H, T, dk = Q.shape
    dv = V.shape[-1]
    if K.shape != Q.shape or V.shape[:3] != Q.shape[:3]:
        raise ValueError(f"shape mismatch q{Q.shape} k{K.shape} v{V.shape}")
    la = np.ascontiguousarray(_f64(log_a).reshape(B, H, T))
    S0a = None if S0 is None else np.ascontiguousarray(_f64(S0).reshape(B, H, dk, dv))
    z0a = None if z0 is None else np.ascontiguousarray(_f64(z0).reshape(B, H, dk))
    O = np.empty((B, H, T, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    rc = (_lib or lib()).oracle_recurrent_gated(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(la), B, H, T, dk, dv, int(bool(phi)),
        _norm_mode(normalize, floor), float(eps), _ptr(S0a), _ptr(z0a), _ptr(O), _ptr(S), _ptr(z))
    if rc != 0:
        raise MemoryError("oracle_recurrent_gated: scratch allocation failed")
    return O, S, z


def recurrent_bwd(q, k, v, gamma, dO, phi: bool = False, normalize: bool = False,
                  eps: float = 1e-6, S0=None, z0=None, dS_T=None, dz_T=None, _lib=None,
                  floor: bool = False, log_a=None):
    """Gradients of ``recurrent`` (or ``recurrent_gated`` with ``log_a``; then
    gamma is ignored) for the loss sum(dO * O) + <dS_T, S_T> + <dz_T, z_T>.

    Returns (dq, dk, dv, dS0, dz0) as float64 arrays of the inputs' shapes.
    """
    Q, K, V = _as4(_f64(q), "q"), _as4(_f64(k), "k"), _as4(_f64(v), "v")
    B, H, T, dk = Q.shape
    dv = V.shape[-1]
    if K.shape != Q.shape or V.shape[:3] != Q.shape[:3]:
        raise ValueError(f"shape mismatch q{Q.shape} k{K.shape} v{V.shape}")
    G = np.ascontiguousarray(_f64(dO).reshape(B, H, T, dv))
    g = None if log_a is not None else np.ascontiguousarray(
        np.broadcast_to(_f64(gamma).reshape(-1), (H,)).astype(np.float64))
    la = None if log_a is None else np.ascontiguousarray(_f64(log_a).reshape(B, H, T))
    S0a = None if S0 is None else np.ascontiguousarray(_f64(S0).reshape(B, H, dk, dv))
    z0a = None if z0 is None else np.ascontiguousarray(_f64(z0).reshape(B, H, dk))
    dSa = None if dS_T is None else np.ascontiguousarray(_f64(dS_T).reshape(B, H, dk, dv))
    dza = None if dz_T is None else np.ascontiguousarray(_f64(dz_T).reshape(B, H, dk))
    dq = np.empty((B, H, T, dk))
    dkk = np.empty((B, H, T, dk))
    dvv = np.empty((B, H, T, dv))
    dS0 = np.empty((B, H, dk, dv))
    dz0 = np.empty((B, H, dk))
    rc = (_lib or lib()).oracle_recurrent_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(g), _ptr(la), B, H, T, dk, dv, int(bool(phi)),
        _norm_mode(normalize, floor), float(eps), _ptr(S0a), _ptr(z0a), _ptr(G), _ptr(dSa),
        _ptr(dza), _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(dS0), _ptr(dz0))
    if rc != 0:
        raise MemoryError("oracle_recurrent_bwd: scratch allocation failed")
    return dq, dkk, dvv, dS0, dz0


def decode_step(q, k, v, gamma, S, z=None, phi: bool = False, normalize: bool = False,
                eps: float = 1e-6, floor: bool = False):
    """One recurrent decode step for [B,H,dk] q,k and [B,H,dv] v.

    Returns (o [B,H,dv], S_new, z_new); the inputs are not modified.
    """
    q4 = _f64(q)[:, :, None, :]
    k4 = _f64(k)[:, :, None, :]
    v4 = _f64(v)[:, :, None, :]
    O, S_new, z_new = recurrent(q4, k4, v4, gamma, phi, normalize, eps, S0=S, z0=z, floor=floor)
    return O[:, :, 0, :], S_new, z_new


def noncausal(q, k, v, phi: bool = False, normalize: bool = False, eps: float = 1e-6,
              _lib=None, floor: bool = False):
    """Non-causal (gamma = 1) form in fp64; returns (O, S, z) like ``recurrent``."""
    Q, K, V = _as4(_f64(q), "q"), _as4(_f64(k), "k"), _as4(_f64(v), "v")
    B, H, T, dk = Q.shape
    dv = V.shape[-1]
    O = np.empty((B, H, T, dv))
    S = np.empty((B, H, dk, dv))
    z = np.empty((B, H, dk))
    rc = (_lib or lib()).oracle_noncausal(
        _ptr(Q), _ptr(K), _ptr(V), B, H, T, dk, dv, int(bool(phi)), _norm_mode(normalize, floor),
        float(eps), _ptr(O), _ptr(S), _ptr(z))
    if rc != 0:
        raise MemoryError("oracle_noncausal: scratch allocation failed")
    return O, S, z


def taylor_features(x, _lib=None):
    """Second-order Taylor features of every row, in fp64: [..., d] -> [..., 1 + d + d^2],
    ordered (1, x, vec(x x^T) / sqrt(2)) with vec row-major ("Linear attention" page,
    box "Taylor features")."""
    X = np.ascontiguousarray(_f64(x))
    d = X.shape[-1]
    n = int(np.prod(X.shape[:-1]))
    out = np.empty(X.shape[:-1] + (1 + d + d * d,))
    (_lib or lib()).oracle_taylor_features(_ptr(X), n, d, _ptr(out))
    return out


def recurrent_taylor(q, k, v, gamma, normalize: bool = False, eps: float = 1e-6, S0=None,
                     z0=None, _lib=None, floor: bool = False):
    """The causal recurrence with the Taylor feature map: ``recurrent`` on the
    features of q and k (d_phi = 1 + d + d^2 rows of S and z, in the order of
    ``taylor_features``).  The page pairs the map with the normaliser, which it
    keeps positive: phi(q)^T phi(k) = ((s + 1)^2 + 1) / 2 >= 1/2."""
    fq, fk = taylor_features(q, _lib), taylor_features(k, _lib)
    return recurrent(fq, fk, v, gamma, phi=False, normalize=normalize, eps=eps, S0=S0, z0=z0,
                     _lib=_lib, floor=floor)


def taylor_features_bwd(x, dfeat, _lib=None):
    """The gradient with respect to x of a loss whose gradient with respect to the
    Taylor features of x is ``dfeat`` ([..., 1 + d + d^2] -> [..., d]): the chain
    rule through (1, x, vec(x x^T) / sqrt(2))."""
    X = np.ascontiguousarray(_f64(x))
    d = X.shape[-1]
    n = int(np.prod(X.shape[:-1]))
    G = np.ascontiguousarray(_f64(dfeat)).reshape(n, 1 + d + d * d)
    out = np.empty(X.shape)
    (_lib or lib()).oracle_taylor_features_bwd(_ptr(X), _ptr(G), n, d, _ptr(out))
    return out


def recurrent_bwd_taylor(q, k, v, gamma, dO, normalize: bool = False, eps: float = 1e-6,
                         S0=None, z0=None, dS_T=None, dz_T=None, _lib=None, floor: bool = False):
    """Gradients of ``recurrent_taylor`` for the loss sum(dO * O) + <dS_T, S_T> +
    <dz_T, z_T>: ``recurrent_bwd`` on the features (phi = identity, d_phi rows),
    then the chain rule through the feature map for q and k.  Returns (dq, dk, dv,
    dS0, dz0); dS0 and dz0 have the features' rows."""
    fq, fk = taylor_features(q, _lib), taylor_features(k, _lib)
    dfq, dfk, dv, dS0, dz0 = recurrent_bwd(fq, fk, v, gamma, dO, phi=False, normalize=normalize,
                                           eps=eps, S0=S0, z0=z0, dS_T=dS_T, dz_T=dz_T,
                                           _lib=_lib, floor=floor)
    return (taylor_features_bwd(q, dfq, _lib), taylor_features_bwd(k, dfk, _lib), dv, dS0, dz0)


def load_mutant(mutant: int, out_dir: str):
    """Load a build of the oracle with a planted mistake (for pin tests only)."""
    return _load(_build.build_mutant(mutant, out_dir))


__all__ = ["recurrent", "recurrent_taylor", "taylor_features", "taylor_features_bwd",
           "recurrent_bwd_taylor", "decode_step", "noncausal",
           "num_threads", "load_mutant", "lib"]
