"""Seeded synthetic inputs for causal decayed linear attention.

This module is the one thing the oracle side (tests, cpu baseline) and the
CUDA side (tests, bench) share.  It holds none of the method's arithmetic:
only the workload table and seeded random numbers.

Recipe (the same for every workload):
  * every tensor is split into independent blocks, one per (b, h) sequence
    (or, for decode inputs, one per step); block ``key`` seeds its own numpy
    ``default_rng([seed, tensor_id, *key])`` stream, so any subset of blocks
    can be regenerated alone and blocks can be drawn on several threads;
  * values are ``standard_normal(dtype=float32)`` times the workload's scale
    (an fp32 multiply), then rounded to the workload dtype with torch's
    round-to-nearest-even ``.to(bfloat16)`` (fp32 workloads keep them);
  * per-head decays are fp32 numbers: fixed lists, the multi-scale schedule
    gamma_h = 1 - 2^(-5-h) (exact in fp32), or uniform draws from stream
    [seed, 99];
  * per-token log decays (workloads with a ``gate``): for each (b, h) a stream
    [seed, 6, b, h] draws u ~ U[0, 2) per token, log a_t = u * log(gamma_h) in
    fp32 (so the mean log decay is the head's log gamma), and one token in 64,
    chosen by a second draw from the same stream, gets log a_t = -8 (a gate that
    nearly resets the state).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

# tensor ids of the keyed streams
Q_ID, K_ID, V_ID = 0, 1, 2
DQ_ID, DK_ID, DV_ID = 3, 4, 5
LOGA_ID = 6
GAMMA_ID = 99

#: The five workloads, then retention with the floored normaliser (xLSTM's
#: max(|q.z|, 1), RetNet's clamped row sums: signed features, decays per head).
#: ``scale_q/k/v`` multiply the N(0,1) draws.
CONFIGS = {
    "tiny_retention_fp32": dict(
        index=0, B=1, H=2, T=256, dk=32, dv=32, dtype="f32", phi=False, normalize=False,
        causal=True, gamma=("list", [0.9, 0.99]), scale_q=32 ** -0.5, scale_k=32 ** -0.5,
        scale_v=32 ** -0.5, seed=0),
    "linear_attention_bf16": dict(
        index=1, B=4, H=8, T=4096, dk=64, dv=64, dtype="bf16", phi=True, normalize=True,
        causal=True, gamma=("list", [1.0] * 8), scale_q=1.0, scale_k=1.0, scale_v=1.0, seed=1),
    "msr_retention_bf16": dict(
        index=2, B=8, H=16, T=8192, dk=128, dv=256, dtype="bf16", phi=False, normalize=False,
        causal=True, gamma=("msr", 16), scale_q=128 ** -0.5, scale_k=128 ** -0.5, scale_v=1.0,
        seed=2),
    "long_retention_bf16": dict(
        index=3, B=1, H=8, T=65536, dk=128, dv=128, dtype="bf16", phi=False, normalize=False,
        causal=True, gamma=("uniform", 0.99, 0.9999), scale_q=128 ** -0.5, scale_k=128 ** -0.5,
        scale_v=128 ** -0.5, seed=3),
    "decode_bf16": dict(
        index=4, B=256, H=32, T=512, dk=128, dv=128, dtype="bf16", phi=False, normalize=False,
        causal=True, gamma=("msr", 8), scale_q=1.0, scale_k=1.0, scale_v=1.0, seed=4,
        decode_steps=1024),
    "retention_floor_bf16": dict(
        index=5, B=4, H=8, T=4096, dk=64, dv=64, dtype="bf16", phi=False, normalize=True,
        floor=True, causal=True, gamma=("msr", 8), scale_q=64 ** -0.5, scale_k=64 ** -0.5,
        scale_v=1.0, seed=5),
    # per-token (gated) decay: the heads' gammas set the mean of the log decays
    "gated_retention_bf16": dict(
        index=6, B=4, H=16, T=4096, dk=128, dv=128, dtype="bf16", phi=False, normalize=False,
        causal=True, gamma=("msr", 8), gate=True, scale_q=128 ** -0.5, scale_k=128 ** -0.5,
        scale_v=1.0, seed=6),
    # the second-order Taylor feature map (Based: q, k projected to d = 16, 1 + 16 + 256 =
    # 273 features), normalised linear attention; q, k ~ N(0, 1/4) so that s = q.k ~ N(0, 1)
    "taylor_linear_attention_bf16": dict(
        index=7, B=8, H=16, T=4096, dk=16, dv=64, dtype="bf16", phi="taylor", normalize=True,
        causal=True, gamma=("list", [1.0] * 16), scale_q=0.5, scale_k=0.5, scale_v=1.0, seed=7),
}

_THREADS = max(1, min(16, (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                           else os.cpu_count() or 1)))


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _block(seed: int, tensor_id: int, key: tuple, shape: tuple, scale: float) -> np.ndarray:
    rng = np.random.default_rng([seed, tensor_id, *key])
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def normal_bhtd(seed: int, tensor_id: int, B: int, H: int, T: int, d: int, scale: float,
                pairs=None) -> np.ndarray:
    """fp32 draws of shape [B,H,T,d], one stream per (b, h).

    With ``pairs`` (a list of (b, h)) only those sequences are drawn and the
    result has shape [len(pairs), T, d]; values equal the full draw's slices.
    """
    keys = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    out = np.empty((len(keys), T, d), dtype=np.float32)

    def work(i):
        b, h = keys[i]
        out[i] = _block(seed, tensor_id, (b, h), (T, d), scale)

    if len(keys) * T * d >= (1 << 20) and _THREADS > 1:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, range(len(keys))))
    else:
        for i in range(len(keys)):
            work(i)
    return out if pairs is not None else out.reshape(B, H, T, d)


def gammas(cfg: dict) -> np.ndarray:
    """Per-head decays as fp32 [H]."""
    H = cfg["H"]
    kind = cfg["gamma"][0]
    if kind == "list":
        g = np.asarray(cfg["gamma"][1], dtype=np.float32)
    elif kind == "msr":  # gamma_h = 1 - 2^(-5 - (h mod period))
        period = cfg["gamma"][1]
        g = np.asarray([1.0 - 2.0 ** (-5 - (h % period)) for h in range(H)], dtype=np.float32)
    elif kind == "uniform":
        lo, hi = cfg["gamma"][1], cfg["gamma"][2]
        g = np.random.default_rng([cfg["seed"], GAMMA_ID]).uniform(lo, hi, H).astype(np.float32)
    else:
        raise ValueError(kind)
    assert g.shape == (H,)
    return g


def log_decays(seed: int, gamma: np.ndarray, B: int, T: int, pairs=None) -> np.ndarray:
    """Per-token log decays [B,H,T] fp32 (or [len(pairs), T]) around the heads'
    gammas; see the module docstring."""
    H = gamma.shape[0]
    keys = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(H)]
    out = np.empty((len(keys), T), dtype=np.float32)
    lg = np.log(gamma.astype(np.float64)).astype(np.float32)
    for i, (b, h) in enumerate(keys):
        rng = np.random.default_rng([seed, LOGA_ID, b, h])
        u = rng.uniform(0.0, 2.0, T).astype(np.float32)
        x = u * lg[h]
        x[rng.integers(0, 64, T) == 0] = np.float32(-8.0)
        out[i] = x
    return out if pairs is not None else out.reshape(B, H, T)


def _to(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(x)
    return t if dtype == "f32" else t.to(torch_dtype(dtype))


def make_inputs(cfg, pairs=None, T=None) -> dict:
    """q, k, v (torch, CPU, workload dtype) and gamma (numpy fp32 [H]).

    ``cfg`` is a CONFIGS key or a dict of the same form.  With ``pairs`` only
    those (b, h) sequences are drawn: q/k/v then have shape [n, T, d] and
    ``gamma_pairs`` holds each one's decay.  ``T`` overrides the length.
    """
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    B, H, dk, dv = c["B"], c["H"], c["dk"], c["dv"]
    T = c["T"] if T is None else T
    s = c["seed"]
    q = normal_bhtd(s, Q_ID, B, H, T, dk, c["scale_q"], pairs)
    k = normal_bhtd(s, K_ID, B, H, T, dk, c["scale_k"], pairs)
    v = normal_bhtd(s, V_ID, B, H, T, dv, c["scale_v"], pairs)
    g = gammas(c)
    out = dict(q=_to(q, c["dtype"]), k=_to(k, c["dtype"]), v=_to(v, c["dtype"]), gamma=g)
    if pairs is not None:
        out["gamma_pairs"] = np.asarray([g[h] for (_, h) in pairs], dtype=np.float32)
    if c.get("gate"):
        out["log_a"] = torch.from_numpy(log_decays(s, g, B, T, pairs))
    return out


def decode_inputs(cfg, step: int, pairs=None) -> dict:
    """q, k ([B,H,dk]) and v ([B,H,dv]) of decode step ``step``; one stream per step.

    With ``pairs`` the full step is drawn and the listed (b, h) rows returned.
    """
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    B, H, dk, dv, s = c["B"], c["H"], c["dk"], c["dv"], c["seed"]
    q = _block(s, DQ_ID, (step,), (B, H, dk), c["scale_q"])
    k = _block(s, DK_ID, (step,), (B, H, dk), c["scale_k"])
    v = _block(s, DV_ID, (step,), (B, H, dv), c["scale_v"])
    if pairs is not None:
        bi = np.asarray([p[0] for p in pairs])
        hi = np.asarray([p[1] for p in pairs])
        q, k, v = q[bi, hi], k[bi, hi], v[bi, hi]
    return dict(q=_to(np.ascontiguousarray(q), c["dtype"]),
                k=_to(np.ascontiguousarray(k), c["dtype"]),
                v=_to(np.ascontiguousarray(v), c["dtype"]))


def decode_inputs_all(cfg, steps: int) -> dict:
    """Every decode step's inputs stacked: q [steps,B,H,dk], k, v (drawn on threads)."""
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    with ThreadPoolExecutor(_THREADS) as ex:
        parts = list(ex.map(lambda st: decode_inputs(c, st), range(steps)))
    return {n: torch.stack([p[n] for p in parts]) for n in ("q", "k", "v")}


def random_case(seed: int, B: int, H: int, T: int, dk: int, dv: int, dtype: str = "f32",
                gamma=None, phi: bool = False, normalize: bool = False, causal: bool = True,
                scale: float | None = None, gate: bool = False) -> dict:
    """A small seeded case in the same recipe, for parity and edge-case tests.

    gamma: None -> H draws from U[0.8, 1.0) (fp32); a float -> that value for
    every head; a list -> those values.  scale defaults to d_k^-1/2 for q, k.
    gate: also draw per-token log decays around those gammas (``log_a``).
    """
    sc = dk ** -0.5 if scale is None else scale
    if gamma is None:
        g = ("list", list(np.random.default_rng([seed, GAMMA_ID]).uniform(0.8, 1.0, H)
                          .astype(np.float32)))
    elif np.isscalar(gamma):
        g = ("list", [float(gamma)] * H)
    else:
        g = ("list", list(gamma))
    cfg = dict(B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, phi=phi, normalize=normalize,
               causal=causal, gamma=g, scale_q=sc, scale_k=sc, scale_v=1.0, seed=seed, gate=gate)
    out = make_inputs(cfg)
    out["cfg"] = cfg
    return out


def sample_pairs(B: int, H: int, n: int, seed: int = 12345) -> list:
    """n distinct (b, h) pairs, always including the first and the last."""
    total = B * H
    n = min(n, total)
    rng = np.random.default_rng([seed, B, H])
    idx = set([0, total - 1])
    while len(idx) < n:
        idx.add(int(rng.integers(0, total)))
    return [(i // H, i % H) for i in sorted(idx)]


def shard_pairs(rank: int, world: int, B: int, H: int) -> list:
    """The (b, h) sequences rank `rank` of `world` owns when each rank runs its own
    batch of B sequences out of a global batch of B * world (weak scaling):
    global batch rows rank*B .. rank*B + B - 1, every head."""
    return [(rank * B + b, h) for b in range(B) for h in range(H)]


def tokens(cfg) -> int:
    c = CONFIGS[cfg] if isinstance(cfg, str) else cfg
    return c["B"] * c["T"]


__all__ = ["CONFIGS", "make_inputs", "decode_inputs", "decode_inputs_all", "random_case",
           "gammas", "log_decays", "sample_pairs", "shard_pairs", "normal_bhtd", "torch_dtype", "tokens"]

