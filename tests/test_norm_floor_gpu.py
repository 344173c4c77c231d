"""The floored normaliser (LA_NORM_FLOOR) on the GPU against the fp64 oracle.

o = phi(q)^T S / max(|phi(q)^T z|, 1): the matrix LSTM's normaliser in the box
"An LSTM whose cell is linear attention" on the "Linear attention" page, equal
to RetNet's division of each score row by the absolute value of its sum clamped
below at 1.  Features here are mostly the identity (signed), so denominators of
both signs and of magnitude below and above 1 occur.  Same metric and
tolerances as the other parity tests.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import pins
import workloads

la = pytest.importorskip("retnet_retention_gb300")

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


def check(name, got, want, tol):
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    err = pins.rel_err(got, want)
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.0e}"


def run(x, phi, causal=True, S0=None, z0=None, path=None, opts=None):
    if path and opts is not None:
        opts.path(path)
    q, k, v = (x[n].to(DEV).contiguous() for n in ("q", "k", "v"))
    B, H, T, dk = q.shape
    O, S, z = la.chunk_fwd(q, k, v, x["gamma"], phi=phi, floor=True, causal=causal, S0=S0, z0=z0,
                           z_out=torch.empty(B, H, dk, device=DEV))
    torch.cuda.synchronize()
    return tuple(t.double().cpu().numpy() for t in (O, S, z))


SHAPES = [  # B, H, T, dk, dv, dtype, path
    (2, 3, 77, 32, 48, "f32", "simt"),
    (1, 2, 300, 64, 64, "f32", "simt"),
    (2, 2, 260, 64, 64, "bf16", "tc"),       # pipelined kernel, tensor-core normaliser
    (1, 2, 200, 128, 128, "bf16", "tc"),     # lockstep kernel (128-wide value block)
    (2, 8, 1000, 128, 128, "bf16", "tc"),    # lockstep, segments folded
    (2, 16, 1000, 64, 64, "bf16", "tc"),     # segments: entry states folded in the output walk
    (1, 1, 3000, 64, 64, "bf16", "tc"),      # segments: scan kernel
]


@pytest.mark.parametrize("phi", [False, True], ids=["identity", "elu1"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_floor_matches_oracle(shape, phi, opts):
    B, H, T, dk, dv, dtype, path = shape
    seed = zlib.crc32(repr((shape, phi, "floor")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype=dtype, scale=0.5)
    O, S, z = run(x, phi, path=path, opts=opts)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=phi, floor=True)
    check("O", O, Or, TOL[dtype])
    check("S_T", S, Sr, TOL[dtype])
    check("z_T", z, zr, TOL[dtype])


def test_floor_is_active_and_inactive_in_the_cases():
    """The inputs the tests use give denominators on both sides of the floor."""
    x = workloads.random_case(5, 2, 2, 260, 64, 64, dtype="bf16", scale=0.5)
    q = x["q"].double().numpy()
    k = x["k"].double().numpy()
    g = np.asarray(x["gamma"], np.float64)
    dens = []
    for b in range(2):
        for h in range(2):
            W = (q[b, h] @ k[b, h].T) * pins.decay_mask(260, g[h])
            dens.append(W.sum(axis=1))
    d = np.abs(np.concatenate(dens))
    assert (d < 1).any() and (d > 1).any()


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_floor_noncausal(path, opts):
    dtype = "f32" if path == "simt" else "bf16"
    x = workloads.random_case(61, 1, 3, 333, 128 if path == "tc" else 32,
                              128 if path == "tc" else 48, dtype=dtype, gamma=1.0, scale=0.3)
    O, S, _ = run(x, False, causal=False, path=path, opts=opts)
    Or, Sr, _ = oracle.noncausal(x["q"], x["k"], x["v"], floor=True)
    check("O", O, Or, TOL[dtype])
    check("S", S, Sr, TOL[dtype])


def test_floor_resume_from_state(opts):
    x = workloads.random_case(62, 2, 16, 1000, 64, 64, dtype="bf16", scale=0.5)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], floor=True)
    t1 = 389
    a = {n: x[n][:, :, :t1].contiguous() for n in ("q", "k", "v")}
    b = {n: x[n][:, :, t1:].contiguous() for n in ("q", "k", "v")}
    a["gamma"] = b["gamma"] = x["gamma"]
    O1, S1, z1 = run(a, False)
    O2, S2, z2 = run(b, False, S0=torch.from_numpy(S1).float().to(DEV),
                     z0=torch.from_numpy(z1).float().to(DEV))
    check("O", np.concatenate([O1, O2], axis=2), Or, TOL["bf16"])
    check("S_T", S2, Sr, TOL["bf16"])
    check("z_T", z2, zr, TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_floor_decode_steps(dtype):
    """Ten decode steps with the floor after a short prefill equal the oracle's
    recurrence over the whole sequence."""
    B, H, T, dk, dv, steps = 3, 4, 40, 64, 32, 10
    x = workloads.random_case(63, B, H, T + steps, dk, dv, dtype=dtype, scale=0.5)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], floor=True)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    _, S, z = la.chunk_fwd(q[:, :, :T].contiguous(), k[:, :, :T].contiguous(),
                           v[:, :, :T].contiguous(), x["gamma"], floor=True,
                           z_out=torch.empty(B, H, dk, device=DEV))
    outs = []
    for t in range(T, T + steps):
        outs.append(la.recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                      v[:, :, t].contiguous(), x["gamma"], S, z, floor=True))
    torch.cuda.synchronize()
    O = torch.stack(outs, dim=2).double().cpu().numpy()
    check("o (decode)", O, Or[:, :, T:], TOL[dtype])
    check("S after decode", S.double().cpu().numpy(), Sr, TOL[dtype])
