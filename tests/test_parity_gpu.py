"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Both sides get the same seeded inputs from ``workloads``; the oracle widens
the exact bf16/fp32 values to fp64.  The error metric is
max|gpu - oracle| / max|oracle| over a whole output tensor, with the
tolerances the method's statement fixes: 1e-4 for fp32 inputs, 2e-2 for
bf16 inputs with fp32 accumulation.

Small cases span several chunks and a ragged tail and run element by
element; the full workloads run on the GPU in the launch configuration the
benchmark times, and the oracle checks every sequence it can afford (all of
them for the prefill workloads, a sample of (b, h) sequences for decode).
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


def to_dev(x):
    return x.to(DEV).contiguous()


def np64(t):
    return t.detach().to("cpu").double().numpy()


def gpu_fwd(case, phi, normalize, causal=True, chunk=0, S0=None, z0=None, eps=1e-6):
    O, S, z = la.chunk_fwd(to_dev(case["q"]), to_dev(case["k"]), to_dev(case["v"]),
                           case["gamma"], phi=phi, normalize=normalize, causal=causal, eps=eps,
                           S0=S0, z0=z0, chunk=chunk,
                           z_out=torch.empty(case["q"].shape[:2] + (case["q"].shape[-1],),
                                             device=DEV))
    torch.cuda.synchronize()
    return np64(O), np64(S), np64(z)


def check(name, got, want, tol):
    err = pins.rel_err(got, want)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.0e}"
    return err


# --------------------------------------------------------------------------- workload 1

def test_tiny_retention_fp32_full():
    c = workloads.CONFIGS["tiny_retention_fp32"]
    x = workloads.make_inputs(c)
    O, S, _ = gpu_fwd(x, False, False)
    Or, Sr, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"])
    check("O", O, Or, TOL["f32"])
    check("S_T", S, Sr, TOL["f32"])


# --------------------------------------------------------------------------- small cases

SHAPES = [  # B, H, T, dk, dv
    (1, 2, 1, 16, 16),
    (2, 3, 37, 32, 48),
    (1, 1, 200, 64, 16),
    (2, 2, 130, 16, 64),
    (1, 2, 257, 128, 256),
    (1, 1, 65, 256, 32),
    (3, 1, 300, 64, 64),
]
FLAGS = [(False, False), (True, True), (True, False)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flags", FLAGS, ids=lambda f: f"phi{int(f[0])}_norm{int(f[1])}")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_causal(shape, flags, dtype):
    B, H, T, dk, dv = shape
    phi, normalize = flags
    seed = zlib.crc32(repr((shape, flags, dtype)).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype=dtype)
    O, S, z = gpu_fwd(x, phi, normalize)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=phi,
                                  normalize=normalize)
    check("O", O, Or, TOL[dtype])
    check("S_T", S, Sr, TOL[dtype])
    check("z_T", z, zr, TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 32, 64, 128])
def test_chunk_size_invariance(chunk, dtype):
    x = workloads.random_case(77, 2, 2, 301, 64, 32, dtype=dtype, gamma=[0.7, 0.97])
    Or, Sr, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"])
    O, S, _ = gpu_fwd(x, False, False, chunk=chunk)
    check(f"O C={chunk}", O, Or, TOL[dtype])
    check(f"S C={chunk}", S, Sr, TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_resume_from_state(dtype):
    """Prefill in two calls (the second starting from the first's state) equals one call."""
    x = workloads.random_case(5, 2, 4, 333, 32, 64, dtype=dtype)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True)
    t1 = 129
    a = {n: x[n][:, :, :t1].contiguous() for n in ("q", "k", "v")}
    b = {n: x[n][:, :, t1:].contiguous() for n in ("q", "k", "v")}
    a["gamma"] = b["gamma"] = x["gamma"]
    O1, S1, z1 = gpu_fwd(a, True, True)
    O2, S2, z2 = gpu_fwd(b, True, True, S0=torch.from_numpy(S1).float().to(DEV),
                         z0=torch.from_numpy(z1).float().to(DEV))
    check("O", np.concatenate([O1, O2], axis=2), Or, TOL[dtype])
    check("S_T", S2, Sr, TOL[dtype])
    check("z_T", z2, zr, TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flags", FLAGS, ids=lambda f: f"phi{int(f[0])}_norm{int(f[1])}")
def test_noncausal(flags, dtype):
    phi, normalize = flags
    x = workloads.random_case(9, 2, 2, 190, 64, 48, dtype=dtype, gamma=1.0)
    O, S, z = gpu_fwd(x, phi, normalize, causal=False)
    Or, Sr, zr = oracle.noncausal(x["q"], x["k"], x["v"], phi=phi, normalize=normalize)
    check("O", O, Or, TOL[dtype])
    check("S", S, Sr, TOL[dtype])
    # the associativity the pages state: Q(K^T V) == (Q K^T) V
    check("left order", O, pins.noncausal_left(np64(x["q"]), np64(x["k"]), np64(x["v"]),
                                               phi=phi, normalize=normalize), TOL[dtype])


@pytest.mark.parametrize("H", [1, 2])
def test_state_walk_with_inputs_just_written(H):
    """Inputs written by a kernel right before each call (still in L2, so the tile
    loads run ahead of the MMAs), segments of two chunks, twelve repeats: the state
    walk's exit state must be read after its last MMA, not an earlier one."""
    B, T, dk, dv = 1, 3000, 64, 64
    x = workloads.random_case(4242 + H, B, H, T, dk, dv, dtype="bf16")
    want_O, want_S, _ = oracle.recurrent(x["q"].flip(2), x["k"].flip(2), x["v"].flip(2), x["gamma"])
    q, k, v = (to_dev(x[n]) for n in ("q", "k", "v"))
    for rep in range(12):
        qf, kf, vf = (t.flip(2).contiguous() for t in (q, k, v))
        O, S, _ = la.chunk_fwd(qf, kf, vf, x["gamma"])
        torch.cuda.synchronize()
        check(f"O (repeat {rep})", np64(O), want_O, TOL["bf16"])
        check(f"S (repeat {rep})", np64(S), want_S, TOL["bf16"])


def test_closed_form_geometric_series():
    """One nonzero feature and value column, q = k = v = 1: o_n = (1 - g^(n+1)) / (1 - g)."""
    T = 65536
    q = torch.zeros(1, 2, T, 16)
    q[..., 0] = 1.0
    v = torch.zeros(1, 2, T, 16)
    v[..., 0] = 1.0
    x = dict(q=q, k=q.clone(), v=v, gamma=np.array([0.99, 0.9999], dtype=np.float32))
    O, S, _ = gpu_fwd(x, False, False)
    n = np.arange(T, dtype=np.float64)
    for h, g in enumerate(x["gamma"].astype(np.float64)):
        want = -np.expm1((n + 1.0) * np.log(g)) / (1.0 - g)
        check(f"gamma={g}", O[0, h, :, 0], want, TOL["f32"])
        assert np.all(O[0, h, :, 1:] == 0.0)


@pytest.mark.parametrize("gated", [False, True], ids=["gamma", "per_token"])
def test_closed_form_past_2_31_elements(gated):
    """Index arithmetic past 2^31 elements: B=64, H=16, T=32768, d=64 in bf16 (each of
    Q, K, V and O holds 2^31 elements, 4 GiB), built on the device.  q = k = e_0 and
    v = c_(b,h) e_0 with a constant per sequence, so o_n = c (1 - g^(n+1)) / (1 - g) for
    the head's gamma (the multi-scale heads' 1 - 2^(-5-h)) and every other column is
    0; a read of another sequence's rows would show as the wrong constant.  Per
    token: the same gamma as a decay at every token (log_a = log gamma), through the
    per-token decay's kernels."""
    B, H, T, d = 64, 16, 32768, 64
    gam = np.array([1.0 - 2.0 ** (-5 - h) for h in range(H)], dtype=np.float32)
    c = (np.arange(B * H).reshape(B, H) % 7 + 1).astype(np.float32)
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device=DEV)
    q[..., 0] = 1.0
    v = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device=DEV)
    v[..., 0] = torch.from_numpy(c).to(DEV, torch.bfloat16)[:, :, None]
    if gated:
        log_a = torch.from_numpy(np.log(gam.astype(np.float64)).astype(np.float32)).to(DEV)
        log_a = log_a[None, :, None].expand(B, H, T).contiguous()
        O, S, _ = la.chunk_fwd(q, q, v, log_a=log_a)
        del log_a
    else:
        O, S, _ = la.chunk_fwd(q, q, v, gam)
    torch.cuda.synchronize()
    del q, v
    assert float(O[..., 1:].float().abs().max()) == 0.0
    got = O[..., 0].double().cpu().numpy()
    del O
    n = np.arange(T, dtype=np.float64)
    g = gam.astype(np.float64)
    geo = -np.expm1((n[None, :] + 1.0) * np.log(g)[:, None]) / (1.0 - g)[:, None]  # [H][T]
    want = c.astype(np.float64)[:, :, None] * geo[None, :, :]
    check("O[..., 0]", got, want, TOL["bf16"])
    # the final state: S[0][0] = c sum_n g^(T-1-n) = c (1 - g^T) / (1 - g), the rest 0
    S_np = S.double().cpu().numpy()
    want_s = c.astype(np.float64) * (-np.expm1(T * np.log(g)) / (1.0 - g))[None, :]
    check("S_T[0, 0]", S_np[:, :, 0, 0], want_s, TOL["bf16"])
    S_np[:, :, 0, 0] = 0.0
    assert np.all(S_np == 0.0)


def test_decode_steps_past_2_31_state_elements():
    """Decode over a state of 2^31 fp32 elements (B=1024, H=128, d_k = d_v = 128; 8 GiB):
    q = k = e_0 and v = c_(b,h) e_0 from S = 0, two steps: o_1 = c, o_2 = c (1 + g)
    in column 0, and S = c (1 + g) e_0 e_0^T; a step on another sequence's state
    block would show as the wrong constant."""
    B, H, d = 1024, 128, 128
    gam = np.array([1.0 - 2.0 ** (-5 - (h % 16)) for h in range(H)], dtype=np.float32)
    c = (np.arange(B * H).reshape(B, H) % 7 + 1).astype(np.float32)
    S = torch.zeros(B, H, d, d, device=DEV)
    q = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
    q[..., 0] = 1.0
    v = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
    v[..., 0] = torch.from_numpy(c).to(DEV, torch.bfloat16)
    o1 = la.recurrent_step(q, q, v, gam, S)
    o2 = la.recurrent_step(q, q, v, gam, S)
    torch.cuda.synchronize()
    g = gam.astype(np.float64)[None, :]
    cc = c.astype(np.float64)
    check("o_1", np64(o1[..., 0]), cc, TOL["bf16"])
    check("o_2", np64(o2[..., 0]), cc * (1.0 + g), TOL["bf16"])
    assert float(o2[..., 1:].float().abs().max()) == 0.0
    check("S[0, 0]", np64(S[:, :, 0, 0]), cc * (1.0 + g), TOL["f32"])
    S[:, :, 0, 0] = 0.0
    assert float(S.abs().max()) == 0.0


def test_empty_sequence_copies_state():
    B, H, dk, dv = 2, 3, 32, 16
    S0 = torch.randn(B, H, dk, dv, device=DEV)
    z0 = torch.randn(B, H, dk, device=DEV)
    e = torch.zeros(B, H, 0, dk, device=DEV)
    O, S, z = la.chunk_fwd(e, e, torch.zeros(B, H, 0, dv, device=DEV), [0.5] * H, S0=S0, z0=z0,
                           normalize=True)
    torch.cuda.synchronize()
    assert O.shape == (B, H, 0, dv)
    assert torch.equal(S, S0) and torch.equal(z, z0)
    O, S, z = la.chunk_fwd(e, e, torch.zeros(B, H, 0, dv, device=DEV), [0.5] * H, normalize=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S) == 0 and torch.count_nonzero(z) == 0


def test_state_init_zeroes():
    S = torch.randn(3, 5, 64, 128, device=DEV)
    z = torch.randn(3, 5, 64, device=DEV)
    la.state_init(S, z)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S) == 0 and torch.count_nonzero(z) == 0


def test_invalid_arguments_on_device():
    q = torch.zeros(1, 1, 8, 16, device=DEV)
    with pytest.raises(la.LinAttnError) as e:
        la.chunk_fwd(q, q, q, [1.5])
    assert e.value.status == la.LA_ERR_INVALID_ARG
    with pytest.raises(la.LinAttnError) as e:
        la.chunk_fwd(q, q, q, [0.5], causal=False)
    assert e.value.status == la.LA_ERR_UNSUPPORTED


# --------------------------------------------------------------------------- decode

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flags", FLAGS, ids=lambda f: f"phi{int(f[0])}_norm{int(f[1])}")
@pytest.mark.parametrize("dims", [(16, 16), (64, 32), (128, 128), (32, 256), (256, 64)])
def test_decode_steps(dims, flags, dtype):
    dk, dv = dims
    phi, normalize = flags
    B, H, T0, steps = 3, 4, 40, 12
    x = workloads.random_case(11, B, H, T0 + steps, dk, dv, dtype=dtype)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=phi,
                                  normalize=normalize)
    q, k, v = (to_dev(x[n]) for n in ("q", "k", "v"))
    _, S, z = la.chunk_fwd(q[:, :, :T0].contiguous(), k[:, :, :T0].contiguous(),
                           v[:, :, :T0].contiguous(), x["gamma"], phi=phi, normalize=normalize,
                           z_out=torch.empty(B, H, dk, device=DEV))
    outs = []
    for t in range(T0, T0 + steps):
        o = la.recurrent_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                              v[:, :, t].contiguous(), x["gamma"], S, z, phi=phi,
                              normalize=normalize)
        outs.append(np64(o))
    torch.cuda.synchronize()
    check("decode o", np.stack(outs, axis=2), Or[:, :, T0:], TOL[dtype])
    check("decode S", np64(S), Sr, TOL[dtype])
    if normalize:
        check("decode z", np64(z), zr, TOL[dtype])


# --------------------------------------------------------------------------- full workloads

def test_linear_attention_bf16_full():
    c = workloads.CONFIGS["linear_attention_bf16"]
    x = workloads.make_inputs(c)
    O, S, z = gpu_fwd(x, True, True)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True)
    check("O", O, Or, TOL["bf16"])
    check("S_T", S, Sr, TOL["bf16"])
    check("z_T", z, zr, TOL["bf16"])


def test_retention_floor_bf16_full():
    """The bench's floored-normaliser workload in the launch configuration the
    bench times (identity features, decays per head, every sequence)."""
    c = workloads.CONFIGS["retention_floor_bf16"]
    x = workloads.make_inputs(c)
    O, S, z = la.chunk_fwd(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), x["gamma"],
                           phi=False, normalize=True, floor=True,
                           z_out=torch.empty(c["B"], c["H"], c["dk"], device=DEV))
    torch.cuda.synchronize()
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], floor=True)
    check("O", np64(O), Or, TOL["bf16"])
    check("S_T", np64(S), Sr, TOL["bf16"])
    check("z_T", np64(z), zr, TOL["bf16"])


def _edge_pairs(B, H, n_pairs):
    """A seeded sample of (b, h) sequences plus the corners of the batch: the last
    batch row and the last head are where the last CTAs of the grid land."""
    return sorted(set(workloads.sample_pairs(B, H, n_pairs)) | {(0, H - 1), (B - 1, 0), (B - 1, H - 1)})


def _sampled_workload(name, n_pairs, causal=True):
    c = workloads.CONFIGS[name]
    x = workloads.make_inputs(c)
    gq = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    pairs = _edge_pairs(c["B"], c["H"], n_pairs)
    O, S, _ = la.chunk_fwd(*gq, x["gamma"], phi=c["phi"], normalize=c["normalize"],
                           causal=causal)
    torch.cuda.synchronize()
    bi = [p[0] for p in pairs]
    hi = [p[1] for p in pairs]
    O_s = O[bi, hi].double().cpu().numpy()
    S_s = S[bi, hi].double().cpu().numpy()
    assert torch.isfinite(O).all() and torch.isfinite(S).all()
    xs = {n: x[n][bi, hi] for n in ("q", "k", "v")}
    g = np.asarray([x["gamma"][h] for h in hi], dtype=np.float32)
    return c, xs, g, O_s, S_s


def test_msr_retention_bf16_full():
    """The multi-scale headline (B8 H16 T8192, d_k 128, d_v 256) in the launch
    configuration the bench times, every output and final state against the oracle;
    the oracle runs one batch row at a time and the errors combine as one
    max|gpu - oracle| / max|oracle| per tensor."""
    c = workloads.CONFIGS["msr_retention_bf16"]
    x = workloads.make_inputs(c)
    O, S, _ = la.chunk_fwd(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), x["gamma"])
    torch.cuda.synchronize()
    err = {"O": 0.0, "S_T": 0.0}
    ref = {"O": 0.0, "S_T": 0.0}
    for b in range(c["B"]):
        Or, Sr, _ = oracle.recurrent(x["q"][b:b + 1], x["k"][b:b + 1], x["v"][b:b + 1], x["gamma"])
        for name, got, want in (("O", O[b:b + 1], Or), ("S_T", S[b:b + 1], Sr)):
            g = np64(got)
            assert np.all(np.isfinite(g)), f"{name}: non-finite output in batch row {b}"
            err[name] = max(err[name], float(np.abs(g - want).max()))
            ref[name] = max(ref[name], float(np.abs(want).max()))
    for name in err:
        rel = err[name] / ref[name]
        assert rel <= TOL["bf16"], f"{name}: rel err {rel:.3e} > {TOL['bf16']:.0e}"


def test_long_retention_bf16_all_heads():
    c, xs, g, O_s, S_s = _sampled_workload("long_retention_bf16", 8)
    Or, Sr, _ = oracle.recurrent(xs["q"][None], xs["k"][None], xs["v"][None], g)
    check("O", O_s, Or[0], TOL["bf16"])
    check("S_T", S_s, Sr[0], TOL["bf16"])


def test_long_retention_noncausal_variant():
    c = dict(workloads.CONFIGS["long_retention_bf16"])
    c["gamma"] = ("list", [1.0] * c["H"])
    x = workloads.make_inputs(c)
    O, S, _ = gpu_fwd(x, False, False, causal=False)
    Or, Sr, _ = oracle.noncausal(x["q"], x["k"], x["v"])
    check("O", O, Or, TOL["bf16"])
    check("S", S, Sr, TOL["bf16"])


def test_decode_bf16_sampled():
    """512-token prefill then 1024 decode steps over B=256, H=32; the oracle follows 6 sequences."""
    name = "decode_bf16"
    c = workloads.CONFIGS[name]
    x = workloads.make_inputs(c)
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    _, S, _ = la.chunk_fwd(q, k, v, x["gamma"])
    del q, k, v
    pairs = _edge_pairs(c["B"], c["H"], 6)
    bi = [p[0] for p in pairs]
    hi = [p[1] for p in pairs]
    steps = c["decode_steps"]
    outs, dq, dk_, dv_ = [], [], [], []
    for t in range(steps):
        d = workloads.decode_inputs(c, t)
        o = la.recurrent_step(to_dev(d["q"]), to_dev(d["k"]), to_dev(d["v"]), x["gamma"], S)
        outs.append(o[bi, hi].double().cpu().numpy())
        dq.append(d["q"][bi, hi])
        dk_.append(d["k"][bi, hi])
        dv_.append(d["v"][bi, hi])
    torch.cuda.synchronize()
    assert torch.isfinite(S).all()
    g = np.asarray([x["gamma"][h] for h in hi], dtype=np.float32)
    # the oracle: prefill then the same steps as one continued recurrence
    qs = torch.cat([x["q"][bi, hi], torch.stack(dq, dim=1)], dim=1)
    ks = torch.cat([x["k"][bi, hi], torch.stack(dk_, dim=1)], dim=1)
    vs = torch.cat([x["v"][bi, hi], torch.stack(dv_, dim=1)], dim=1)
    Or, Sr, _ = oracle.recurrent(qs[None], ks[None], vs[None], g)
    check("decode outputs", np.stack(outs, axis=1), Or[0, :, c["T"]:], TOL["bf16"])
    check("final state", S[bi, hi].double().cpu().numpy(), Sr[0], TOL["bf16"])


@pytest.mark.parametrize("pieces", [1, 2, 3])
def test_host_entry_point_pipelined(pieces):
    """chunk_fwd_host: pinned host inputs in, host results out, batch split over
    two side streams; equals the oracle (initial state included)."""
    x = workloads.random_case(91, 3, 2, 300, 64, 64, dtype="bf16")
    rng = np.random.default_rng(5)
    S0 = torch.from_numpy(rng.standard_normal((3, 2, 64, 64)).astype(np.float32) * 0.1)
    z0 = torch.from_numpy(np.abs(rng.standard_normal((3, 2, 64))).astype(np.float32))
    times = []
    O, S, z = la.chunk_fwd_host(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(),
                                x["gamma"], phi=True, normalize=True, S0=S0.pin_memory(),
                                z0=z0.pin_memory(), pieces=pieces, timing=times)
    assert O.device.type == "cpu" and len(times) == 1 and times[0] > 0
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True,
                                  S0=S0, z0=z0)
    check("O", np64(O), Or, TOL["bf16"])
    check("S_T", np64(S), Sr, TOL["bf16"])
    check("z_T", np64(z), zr, TOL["bf16"])


def test_host_entry_point_plain_retention_segments():
    """la_chunk_fwd_host on plain retention (the factored-decay build) with few
    sequences, so each piece's plan cuts its sequences into segments."""
    x = workloads.random_case(93, 2, 2, 3000, 128, 128, dtype="bf16")
    O, S, _ = la.chunk_fwd_host(x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory(),
                                x["gamma"], pieces=2)
    Or, Sr, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"])
    check("O", np64(O), Or, TOL["bf16"])
    check("S_T", np64(S), Sr, TOL["bf16"])
