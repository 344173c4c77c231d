"""The Taylor feature map (LA_PHI_TAYLOR) on the GPU against the fp64 oracle.

The kernel builds phi(x) = (1, x, vec(x x^T)/sqrt 2) of the 16-wide queries and
keys on chip (273 features); the oracle expands them in fp64 ("Linear attention"
page, box "Taylor features") and runs the plain recurrence.  Shapes span one
chunk and several, ragged tails, two value blocks, per-head decays and gamma = 1,
with and without the normaliser, with an initial state, and the final state in
the page's feature order.  Same metric and bf16 tolerance as the other parity
tests: max|gpu - oracle| / max|oracle| <= 2e-2.
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

TOL = 2e-2
DEV = "cuda"
DF = 273


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


def check(name, got, want, tol=TOL):
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    err = pins.rel_err(got, want)
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.0e}"


def np64(t):
    return t.detach().to("cpu").double().numpy()


def case(shape, gamma, seed_tag):
    B, H, T, dv = shape
    seed = zlib.crc32(repr((shape, gamma, seed_tag)).encode()) % 100000
    return workloads.random_case(seed, B, H, T, 16, dv, dtype="bf16", gamma=gamma, scale=0.5)


SHAPES = [  # B, H, T, d_v
    (1, 2, 1, 64),
    (1, 2, 77, 64),
    (2, 2, 128, 64),
    (2, 3, 300, 64),
    (1, 2, 260, 128),
    (1, 1, 1000, 64),
]


@pytest.mark.parametrize("normalize", [True, False], ids=["normalised", "plain"])
@pytest.mark.parametrize("gamma", [None, 1.0], ids=["decayed", "gamma1"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_taylor_matches_oracle(shape, gamma, normalize):
    x = case(shape, gamma, "taylor")
    B, H, T, dv = shape
    O, S, z = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"],
                           phi="taylor", normalize=normalize,
                           z_out=torch.empty((B, H, DF), device=DEV))
    torch.cuda.synchronize()
    assert S.shape == (B, H, DF, dv) and z.shape == (B, H, DF)
    Or, Sr, zr = oracle.recurrent_taylor(x["q"], x["k"], x["v"], x["gamma"], normalize=normalize)
    check("O", np64(O), Or)
    check("S_T", np64(S), Sr)
    check("z_T", np64(z), zr)


@pytest.mark.parametrize("normalize", [True, False], ids=["normalised", "plain"])
def test_taylor_from_an_initial_state(normalize):
    """A chunked call resumed from the state of the first part equals one pass; the
    initial state enters in the page's feature order."""
    B, H, T, dv = 2, 2, 400, 64
    x = case((B, H, T, dv), None, "resume")
    rng = np.random.default_rng(5)
    S0 = torch.from_numpy(rng.standard_normal((B, H, DF, dv)).astype(np.float32) * 0.1)
    z0 = torch.from_numpy(np.abs(rng.standard_normal((B, H, DF))).astype(np.float32) + 1.0)
    O, S, z = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"],
                           phi="taylor", normalize=normalize, S0=S0.to(DEV), z0=z0.to(DEV),
                           z_out=torch.empty((B, H, DF), device=DEV))
    torch.cuda.synchronize()
    Or, Sr, zr = oracle.recurrent_taylor(x["q"], x["k"], x["v"], x["gamma"], normalize=normalize,
                                         S0=S0, z0=z0)
    check("O", np64(O), Or)
    check("S_T", np64(S), Sr)
    check("z_T", np64(z), zr)
    # split at a chunk boundary and at a ragged point: the second part starts from the first's state
    for cut in (128, 201):
        q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
        O1, S1, z1 = la.chunk_fwd(q[:, :, :cut].contiguous(), k[:, :, :cut].contiguous(),
                                  v[:, :, :cut].contiguous(), x["gamma"], phi="taylor",
                                  normalize=normalize, S0=S0.to(DEV), z0=z0.to(DEV),
                                  z_out=torch.empty((B, H, DF), device=DEV))
        O2, S2, _ = la.chunk_fwd(q[:, :, cut:].contiguous(), k[:, :, cut:].contiguous(),
                                 v[:, :, cut:].contiguous(), x["gamma"], phi="taylor",
                                 normalize=normalize, S0=S1, z0=z1)
        torch.cuda.synchronize()
        check(f"O split at {cut}", np.concatenate([np64(O1), np64(O2)], axis=2), Or)
        check(f"S_T split at {cut}", np64(S2), Sr)


def test_taylor_empty_sequence_copies_the_state():
    B, H, dv = 1, 2, 64
    S0 = torch.randn(B, H, DF, dv, device=DEV)
    q = torch.empty((B, H, 0, 16), dtype=torch.bfloat16, device=DEV)
    v = torch.empty((B, H, 0, dv), dtype=torch.bfloat16, device=DEV)
    _, S, _ = la.chunk_fwd(q, q, v, [0.9, 0.95], phi="taylor", S0=S0)
    torch.cuda.synchronize()
    assert torch.equal(S, S0)


def test_taylor_normalised_constant_values_return_unchanged():
    """With the normaliser the outputs are convex combinations of the v rows (the
    kernel is >= 1/2 > 0), so a constant V comes back unchanged."""
    B, H, T, dv = 1, 2, 700, 64
    x = case((B, H, T, dv), None, "const")
    v = torch.full((B, H, T, dv), 0.375, dtype=torch.bfloat16)
    O, _, _ = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), v.to(DEV), x["gamma"], phi="taylor",
                           normalize=True)
    torch.cuda.synchronize()
    np.testing.assert_allclose(np64(O), 0.375, rtol=1e-2)


def test_taylor_timeout_is_reported_not_hung(opts):
    opts.force_timeout(True)
    x = case((1, 2, 256, 64), None, "timeout")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"], phi="taylor",
                 dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == la.LA_ERR_TIMEOUT
    opts.force_timeout(False)
    status.zero_()
    O, _, _ = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"],
                           phi="taylor", dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Or, _, _ = oracle.recurrent_taylor(x["q"], x["k"], x["v"], x["gamma"])
    check("O after a reported timeout", np64(O), Or)


def test_taylor_linear_attention_bf16_full():
    """The Taylor workload at full size (B=8 H=16 T=4096, d=16 -> 273 features,
    d_v=64, normalised, gamma = 1) in the launch the benchmark times, every sequence
    against the oracle (one batch row at a time; the errors combine as one
    max|gpu - oracle| / max|oracle| per tensor)."""
    c = workloads.CONFIGS["taylor_linear_attention_bf16"]
    x = workloads.make_inputs(c)
    B = c["B"]
    O, S, z = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"],
                           phi="taylor", normalize=True)
    torch.cuda.synchronize()
    err = {"O": 0.0, "S_T": 0.0, "z_T": 0.0}
    ref = dict(err)
    for b in range(B):
        sl = lambda t: t[b:b + 1]
        Or, Sr, zr = oracle.recurrent_taylor(sl(x["q"]), sl(x["k"]), sl(x["v"]), x["gamma"],
                                             normalize=True)
        for name, got, want in (("O", O[b:b + 1], Or), ("S_T", S[b:b + 1], Sr), ("z_T", z[b:b + 1], zr)):
            g = np64(got)
            assert np.all(np.isfinite(g)), f"{name}: non-finite output in batch row {b}"
            err[name] = max(err[name], float(np.abs(g - want).max()))
            ref[name] = max(ref[name], float(np.abs(want).max()))
    for name in err:
        rel = err[name] / ref[name]
        assert rel <= 2e-2, f"{name}: rel err {rel:.3e} > 2e-02"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("normalize", [True, False], ids=["normalised", "plain"])
@pytest.mark.parametrize("dv", [64, 128])
def test_taylor_decode_steps(dv, normalize, dtype):
    """Decode steps with the Taylor map (la_recurrent_step with LA_PHI_TAYLOR): the
    273-row state updated in place, against the oracle's recurrence one token at a
    time from a random initial state in the page's feature order."""
    B, H, steps = 2, 3, 5
    x = workloads.random_case(31 + dv, B, H, steps, 16, dv, dtype=dtype, scale=0.5)
    rng = np.random.default_rng(dv)
    S = torch.from_numpy(rng.standard_normal((B, H, DF, dv)).astype(np.float32) * 0.1)
    z = torch.from_numpy(np.abs(rng.standard_normal((B, H, DF))).astype(np.float32) + 1.0)
    Sd, zd = S.to(DEV), z.to(DEV)
    Sr, zr = S.double().numpy(), z.double().numpy()
    tol = 1e-4 if dtype == "f32" else TOL
    for t in range(steps):
        q, k, v = (x[n][:, :, t].contiguous() for n in ("q", "k", "v"))
        o = la.recurrent_step(q.to(DEV), k.to(DEV), v.to(DEV), x["gamma"], Sd,
                              zd if normalize else None, phi="taylor", normalize=normalize)
        torch.cuda.synchronize()
        Or, Sr, zr = oracle.recurrent_taylor(q[:, :, None], k[:, :, None], v[:, :, None], x["gamma"],
                                             normalize=normalize, S0=Sr,
                                             z0=zr if normalize else None)
        check(f"o step {t}", np64(o), Or[:, :, 0], tol)
        check(f"S step {t}", np64(Sd), Sr, tol)
        if normalize:
            check(f"z step {t}", np64(zd), zr, tol)


def test_taylor_prefill_then_decode_equals_one_prefill():
    """The chunkwise prefill's final state (the kernel's symmetric coordinates
    turned back into the page's order) carries on in the decode step exactly as one
    longer prefill would."""
    B, H, T, dv, extra = 1, 2, 300, 64, 3
    x = case((B, H, T + extra, dv), None, "prefill-decode")
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    _, S, z = la.chunk_fwd(q[:, :, :T].contiguous(), k[:, :, :T].contiguous(), v[:, :, :T].contiguous(),
                           x["gamma"], phi="taylor", normalize=True)
    outs = []
    for t in range(T, T + extra):
        outs.append(la.recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                      v[:, :, t].contiguous(), x["gamma"], S, z, phi="taylor",
                                      normalize=True))
    torch.cuda.synchronize()
    Or, Sr, _ = oracle.recurrent_taylor(x["q"], x["k"], x["v"], x["gamma"], normalize=True)
    check("decoded outputs", np.stack([np64(o) for o in outs], axis=2), Or[:, :, T:])
    check("final state", np64(S), Sr)


def test_taylor_with_the_floored_normaliser():
    """LA_PHI_TAYLOR with LA_NORM_FLOOR: divide by max(|phi(q)^T z|, 1), chunkwise and
    in the decode step (the Taylor kernel is >= 1/2, so short prefixes with gamma < 1
    sit below the floor)."""
    B, H, T, dv = 1, 2, 300, 64
    x = case((B, H, T, dv), [0.3, 0.5], "floor")
    O, S, z = la.chunk_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["gamma"], phi="taylor",
                           floor=True)
    torch.cuda.synchronize()
    Or, Sr, zr = oracle.recurrent_taylor(x["q"], x["k"], x["v"], x["gamma"], floor=True)
    check("O", np64(O), Or)
    check("S_T", np64(S), Sr)
    check("z_T", np64(z), zr)
    q1, k1, v1 = (workloads.random_case(77, B, H, 1, 16, dv, dtype="bf16", scale=0.5)[n][:, :, 0].contiguous()
                  for n in ("q", "k", "v"))
    o = la.recurrent_step(q1.to(DEV), k1.to(DEV), v1.to(DEV), x["gamma"], S, z, phi="taylor", floor=True)
    torch.cuda.synchronize()
    Or1, Sr1, _ = oracle.recurrent_taylor(q1[:, :, None], k1[:, :, None], v1[:, :, None], x["gamma"],
                                          floor=True, S0=Sr, z0=zr)
    check("decode o", np64(o), Or1[:, :, 0])
    check("decode S", np64(S), Sr1)


BWD_SHAPES = [  # B, H, T, d_v, dtype
    (1, 2, 1, 64, "bf16"),
    (1, 2, 100, 64, "bf16"),
    (2, 1, 300, 32, "f32"),
    (1, 1, 1000, 64, "bf16"),  # segments of the backward sweeps
]


@pytest.mark.parametrize("normalize", [True, False], ids=["normalised", "plain"])
@pytest.mark.parametrize("gamma", [1.0, None], ids=["gamma1", "decay"])
@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_taylor_bwd_matches_oracle(shape, gamma, normalize):
    """la_chunk_bwd with the Taylor map (the features built in shared memory, their
    gradients taken back to 16 columns through the map's transpose Jacobian) against
    the oracle's gradients of the recurrence with the map, with an initial state and
    final-state gradients in the features' order."""
    B, H, T, dv, dtype = shape
    seed = zlib.crc32(repr((shape, gamma, normalize, "taylor-bwd")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, 16, dv, dtype=dtype, gamma=gamma, scale=0.5)
    rng = np.random.default_rng(seed)
    tdt = workloads.torch_dtype(dtype)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(tdt)
    S0 = torch.from_numpy(rng.standard_normal((B, H, DF, dv)).astype(np.float32) * 0.05)
    z0 = torch.from_numpy(np.abs(rng.standard_normal((B, H, DF))).astype(np.float32) * 0.1 + 0.5)
    dST = torch.from_numpy(rng.standard_normal((B, H, DF, dv)).astype(np.float32) * 0.05)
    dzT = torch.from_numpy(rng.standard_normal((B, H, DF)).astype(np.float32) * 0.05)
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    dq, dk, dv_, dS0, dz0 = la.chunk_bwd(
        q, k, v, g_o, x["gamma"], phi="taylor", normalize=normalize, S0=S0.to(DEV),
        z0=z0.to(DEV) if normalize else None, dS_T=dST.to(DEV),
        dz_T=dzT.to(DEV) if normalize else None)
    torch.cuda.synchronize()
    rq, rk, rv, rS0, rz0 = oracle.recurrent_bwd_taylor(
        x["q"], x["k"], x["v"], x["gamma"], dO, normalize=normalize, S0=S0,
        z0=z0 if normalize else None, dS_T=dST, dz_T=dzT if normalize else None)
    tol = 1e-4 if dtype == "f32" else TOL
    check("dq", np64(dq), rq, tol)
    check("dk", np64(dk), rk, tol)
    check("dv", np64(dv_), rv, tol)
    check("dS0", np64(dS0), rS0, tol)
    if normalize:
        check("dz0", np64(dz0), rz0, tol)
