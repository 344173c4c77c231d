"""Per-token (gated) decay on the GPU against the fp64 oracle.

S_t = a_t S_{t-1} + phi(k_t) v_t^T with a_t = e^(log_a[b, h, t]): the generic
"decay the old state, add, read out" loop of "Linear Attention, RWKV, and
RetNet" (temporalbook 13.3, subsection 4) with the gate G_t = a_t 1 of "Gated
Linear Attention" (temporalbook 12.5).  The decays come from the workloads
recipe: around each head's gamma, with a near-reset (a = e^-8) every 64 tokens
on average.  Shapes cover the pipelined kernel's widths (64-wide value blocks
for d_k = 128 and for the normaliser), ragged tails, segments folded in the
output walk and segments through the scan kernel, and the CUDA-core kernel in
fp32 and bf16.  Same metric and tolerances as the other parity tests.
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


def run(x, phi=False, normalize=False, floor=False, S0=None, z0=None):
    q, k, v = (x[n].to(DEV).contiguous() for n in ("q", "k", "v"))
    B, H, T, dk = q.shape
    O, S, z = la.chunk_fwd(q, k, v, log_a=x["log_a"].to(DEV).contiguous(), phi=phi,
                           normalize=normalize, floor=floor, S0=S0, z0=z0,
                           z_out=torch.empty(B, H, dk, device=DEV))
    torch.cuda.synchronize()
    return tuple(t.double().cpu().numpy() for t in (O, S, z))


SHAPES = [  # B, H, T, dk, dv, dtype, path
    (2, 3, 77, 32, 48, "f32", "simt"),
    (1, 2, 300, 64, 64, "f32", "simt"),
    (1, 2, 200, 64, 64, "bf16", "simt"),
    (2, 2, 260, 64, 64, "bf16", "tc"),
    (1, 3, 300, 128, 128, "bf16", "tc"),      # d_k = 128: two 64-wide value blocks
    (2, 1, 129, 64, 128, "bf16", "tc"),
    (1, 2, 517, 128, 256, "bf16", "tc"),
    (2, 16, 1000, 64, 64, "bf16", "tc"),      # segments folded in the output walk
    (1, 1, 3000, 64, 64, "bf16", "tc"),       # segments through the scan kernel
    (1, 2, 4100, 128, 128, "bf16", "tc"),     # scan, d_k = 128
]
FLAGS = [(False, False, False), (True, True, False), (False, False, True)]


@pytest.mark.parametrize("flags", FLAGS, ids=["plain", "phi_norm", "floor"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gated_matches_oracle(shape, flags, opts):
    B, H, T, dk, dv, dtype, path = shape
    phi, normalize, floor = flags
    opts.path(path)
    seed = zlib.crc32(repr((shape, flags, "gated")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype=dtype, gate=True,
                              scale=0.5 if floor else None)
    O, S, z = run(x, phi, normalize, floor)
    Or, Sr, zr = oracle.recurrent_gated(x["q"], x["k"], x["v"], x["log_a"], phi=phi,
                                        normalize=normalize, floor=floor)
    check("O", O, Or, TOL[dtype])
    check("S_T", S, Sr, TOL[dtype])
    check("z_T", z, zr, TOL[dtype])


def test_gated_launch_count_follows_the_plan(opts):
    """The decays' prep kernel, then the state walk, [scan,] output walk."""
    opts.path("tc")
    lib = la.library()
    assert lib.la_chunk_fwd_launches(2, 16, 1000, 64, 64, 1, la.LA_GATED, 0) == 3
    assert lib.la_chunk_fwd_launches(1, 1, 3000, 64, 64, 1, la.LA_GATED, 0) == 4
    assert lib.la_chunk_fwd_launches(4, 16, 4096, 128, 128, 1, la.LA_GATED, 0) == 2
    x = workloads.random_case(5, 1, 1, 3000, 64, 64, dtype="bf16", gate=True)
    la.trace_enable(64)
    try:
        run(x)
        names = [n for n, _ in la.trace_collect()]
    finally:
        la.trace_enable(0)
    assert names[0] == "gate_prep_kernel" and names[-1].endswith("/full"), names
    assert len(names) == 4, names


def test_gated_resume_from_state(opts):
    """A split prefill (segments folded) continued from the first part's state."""
    opts.path("tc")
    x = workloads.random_case(7, 2, 16, 1000, 64, 64, dtype="bf16", gate=True)
    Or, Sr, zr = oracle.recurrent_gated(x["q"], x["k"], x["v"], x["log_a"], phi=True,
                                        normalize=True)
    t1 = 389
    a = {n: x[n][:, :, :t1].contiguous() for n in ("q", "k", "v", "log_a")}
    b = {n: x[n][:, :, t1:].contiguous() for n in ("q", "k", "v", "log_a")}
    O1, S1, z1 = run(a, True, True)
    O2, S2, z2 = run(b, True, True, S0=torch.from_numpy(S1).float().to(DEV),
                     z0=torch.from_numpy(z1).float().to(DEV))
    check("O", np.concatenate([O1, O2], axis=2), Or, TOL["bf16"])
    check("S_T", S2, Sr, TOL["bf16"])
    check("z_T", z2, zr, TOL["bf16"])


def test_constant_gate_equals_gamma(opts):
    """log a_t = log gamma_h for every token gives the per-head decay's results
    (two different kernel builds)."""
    opts.path("tc")
    x = workloads.random_case(9, 2, 4, 700, 64, 64, dtype="bf16")
    B, H, T = 2, 4, 700
    lg = np.log(np.asarray(x["gamma"], np.float64)).astype(np.float32)
    x["log_a"] = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(lg[None, :, None], (B, H, T))))
    Og, Sg, _ = run(x)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    O, S, _ = la.chunk_fwd(q, k, v, x["gamma"])
    torch.cuda.synchronize()
    check("O", Og, O.double().cpu().numpy(), TOL["bf16"])
    check("S_T", Sg, S.double().cpu().numpy(), TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_decode_steps(dtype):
    """Decode steps with per-token decays after a gated prefill equal the oracle's
    recurrence over the whole sequence."""
    B, H, T, dk, dv, steps = 3, 4, 40, 64, 32, 10
    x = workloads.random_case(11, B, H, T + steps, dk, dv, dtype=dtype, gate=True)
    Or, Sr, zr = oracle.recurrent_gated(x["q"], x["k"], x["v"], x["log_a"], phi=True,
                                        normalize=True)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    lg = x["log_a"].to(DEV)
    _, S, z = la.chunk_fwd(q[:, :, :T].contiguous(), k[:, :, :T].contiguous(),
                           v[:, :, :T].contiguous(), log_a=lg[:, :, :T].contiguous(), phi=True,
                           normalize=True, z_out=torch.empty(B, H, dk, device=DEV))
    outs = []
    for t in range(T, T + steps):
        outs.append(la.recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                      v[:, :, t].contiguous(), None, S, z, phi=True,
                                      normalize=True, log_a=lg[:, :, t].contiguous()))
    torch.cuda.synchronize()
    O = torch.stack(outs, dim=2).double().cpu().numpy()
    check("o (decode)", O, Or[:, :, T:], TOL[dtype])
    check("S after decode", S.double().cpu().numpy(), Sr, TOL[dtype])
    check("z after decode", z.double().cpu().numpy(), zr, TOL[dtype])


def test_gated_retention_bf16_full():
    """The bench's gated workload in the bench's launch configuration (the output
    walk's CTAs picking the factored body or the row scalings), every sequence
    against the oracle."""
    c = workloads.CONFIGS["gated_retention_bf16"]
    x = workloads.make_inputs(c)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    O, S, _ = la.chunk_fwd(q, k, v, log_a=x["log_a"].to(DEV))
    torch.cuda.synchronize()
    Or, Sr, _ = oracle.recurrent_gated(x["q"], x["k"], x["v"], x["log_a"])
    check("O", O.double().cpu().numpy(), Or, TOL["bf16"])
    check("S_T", S.double().cpu().numpy(), Sr, TOL["bf16"])


SPLIT_CASES = [  # B, H, T, dk, dv: per-token decay, no normaliser, no z
    (2, 16, 1000, 64, 64),   # segments folded in the output walk
    (1, 1, 3000, 64, 64),    # segments with a scan
    (4, 4, 300, 128, 128),   # one segment, 64-wide value blocks
    (2, 3, 200, 64, 128),
    (1, 2, 129, 64, 64),     # one full chunk and a one-row chunk
]


@pytest.mark.parametrize("strong", [0.3, 0.43, 0.6], ids=["a0.3", "a0.43", "a0.6"])
@pytest.mark.parametrize("shape", SPLIT_CASES, ids=lambda s: "x".join(map(str, s)))
def test_gated_factored_and_row_scaled_builds(shape, strong, opts):
    """Per-token decay without normaliser or z: each CTA of the output walk picks the
    factored build when its sequence's chunks all keep their decay from first row to
    last at or above 2^-160, else the row scalings.  Every other
    sequence here decays strongly: a_t around 0.3 (about 2^-220 over a chunk: row
    scalings), 0.43 (about 2^-155, chunks on both sides of the bound: factors up to
    2^+-80 in the factored build) or 0.6 (about 2^-94: factors near 2^+-47 about the
    chunk's middle); the rest follow the recipe's gates.  Outputs and final states
    are checked against the oracle, and the trace against the launch count."""
    opts.path("tc")
    B, H, T, dk, dv = shape
    x = workloads.random_case(zlib.crc32(repr((shape, strong)).encode()) % 100000, B, H, T, dk, dv,
                              dtype="bf16", gate=True)
    log_a = x["log_a"].clone()
    sel = torch.zeros(B * H, dtype=torch.bool)
    sel[::2] = True
    sel = sel.view(B, H)
    log_a[sel] = float(np.log(strong)) + 0.05 * log_a[sel]
    q, k, v = (x[n].to(DEV).contiguous() for n in ("q", "k", "v"))
    la.trace_enable(256)
    try:
        la.trace_collect()
        O, S, _ = la.chunk_fwd(q, k, v, log_a=log_a.to(DEV).contiguous())
        torch.cuda.synchronize()
        names = [n for n, _ in la.trace_collect()]
    finally:
        la.trace_enable(0)
    assert len(names) == la.library().la_chunk_fwd_launches(B, H, T, dk, dv, 1, la.LA_GATED, 0), names
    assert sum(n == "chunk_tc_ws_kernel/full" for n in names) == 1, names
    Or, Sr, _ = oracle.recurrent_gated(x["q"], x["k"], x["v"], log_a)
    check("O", O.double().cpu().numpy(), Or, TOL["bf16"])
    check("S_T", S.double().cpu().numpy(), Sr, TOL["bf16"])
