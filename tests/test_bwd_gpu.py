"""The backward pass (la_chunk_bwd) on the GPU against the fp64 oracle.

The loss is L = sum(dO * O) + <dS_T, S_T> + <dz_T, z_T>; the gradients of Q,
K, V and of the initial state are compared with the oracle's two sweeps of
cumulative sums ("Linear attention" page, "Decoding, training, and what each
costs"), which are themselves pinned by central differences.  Shapes cover one
and several chunks, ragged tails, d_k != d_v, the widest supported state (128 x
128), phi with the normaliser, the floored normaliser, per-head and per-token
decays, and an initial state with a final-state gradient.  Same metric and
tolerances as the forward parity tests.
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


def to_np(t):
    return t.double().cpu().numpy()


SHAPES = [  # B, H, T, dk, dv, dtype
    (1, 2, 1, 16, 16, "f32"),
    (2, 3, 77, 32, 48, "f32"),
    (1, 2, 300, 64, 64, "f32"),
    (2, 2, 260, 64, 64, "bf16"),
    (1, 2, 130, 128, 128, "bf16"),
    (2, 1, 97, 64, 128, "bf16"),
    (1, 1, 1000, 64, 64, "bf16"),  # 16 segments of two chunks, the last one ragged
]
FLAGS = [(False, False, False), (True, True, False), (False, False, True)]


@pytest.mark.parametrize("gated", [False, True], ids=["gamma", "gated"])
@pytest.mark.parametrize("flags", FLAGS, ids=["plain", "phi_norm", "floor"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_matches_oracle(shape, flags, gated):
    B, H, T, dk, dv, dtype = shape
    phi, normalize, floor = flags
    seed = zlib.crc32(repr((shape, flags, gated, "bwd")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype=dtype, gate=gated,
                              scale=0.5 if floor else None)
    rng = np.random.default_rng(seed)
    tdt = workloads.torch_dtype(dtype)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(tdt)
    S0 = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.3)
    z0 = torch.from_numpy(np.abs(rng.standard_normal((B, H, dk))).astype(np.float32))
    dST = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.1)
    dzT = torch.from_numpy(rng.standard_normal((B, H, dk)).astype(np.float32) * 0.1)
    norm_any = normalize or floor
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    kw = dict(log_a=x["log_a"].to(DEV)) if gated else dict(gamma=x["gamma"])
    dq, dk_, dv_, dS0, dz0 = la.chunk_bwd(
        q, k, v, g_o, phi=phi, normalize=normalize, floor=floor, S0=S0.to(DEV),
        z0=z0.to(DEV) if norm_any else None, dS_T=dST.to(DEV), dz_T=dzT.to(DEV) if norm_any else None,
        **kw)
    torch.cuda.synchronize()
    rq, rk, rv, rS0, rz0 = oracle.recurrent_bwd(
        x["q"], x["k"], x["v"], x["gamma"], dO, phi=phi, normalize=normalize, floor=floor,
        S0=S0, z0=z0 if norm_any else None, dS_T=dST, dz_T=dzT if norm_any else None,
        log_a=x["log_a"] if gated else None)
    tol = TOL[dtype]
    check("dq", to_np(dq), rq, tol)
    check("dk", to_np(dk_), rk, tol)
    check("dv", to_np(dv_), rv, tol)
    check("dS0", to_np(dS0), rS0, tol)
    if norm_any:
        check("dz0", to_np(dz0), rz0, tol)


TC_SHAPES = [  # B, H, T, dk, dv: bf16, per-head decay, no phi, no normaliser
    (2, 2, 260, 64, 64),
    (1, 2, 130, 128, 128),
    (2, 1, 97, 64, 128),
    (1, 3, 300, 128, 64),
    (1, 2, 3000, 64, 64),     # the forward passes split into segments (scan)
    (2, 16, 1000, 64, 64),    # segments folded in the output walk
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bwd_tensor_core_path(shape, opts):
    """The three forward passes on the tensor cores (dQ; dV and dK in reversed time,
    walked backward by the kernel itself for these gammas) against the oracle, with an
    initial state and a final-state gradient."""
    opts.path("auto")
    B, H, T, dk, dv = shape
    seed = zlib.crc32(repr((shape, "bwd-tc")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16")
    rng = np.random.default_rng(seed)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    S0 = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.3)
    dST = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.1)
    lib = la.library()
    need = lib.la_bwd_workspace_size(B, H, T, dk, dv, 1, 0)
    assert need > B * H * T * (dk + dv) * 2  # the reversed copies: the tensor-core path
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    dq, dk_, dv_, dS0, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], S0=S0.to(DEV), dS_T=dST.to(DEV))
    torch.cuda.synchronize()
    rq, rk, rv, rS0, _ = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO, S0=S0,
                                              dS_T=dST)
    check("dq", to_np(dq), rq, TOL["bf16"])
    check("dk", to_np(dk_), rk, TOL["bf16"])
    check("dv", to_np(dv_), rv, TOL["bf16"])
    check("dS0", to_np(dS0), rS0, TOL["bf16"])
    # the same through the CUDA-core kernel
    opts.path("simt")
    sq, sk, sv, sS0, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], S0=S0.to(DEV), dS_T=dST.to(DEV))
    torch.cuda.synchronize()
    check("dq tc vs simt", to_np(dq), to_np(sq), TOL["bf16"])
    check("dS0 tc vs simt", to_np(dS0), to_np(sS0), TOL["bf16"])


@pytest.mark.parametrize("shape,gammas", [((2, 2, 260, 64, 64), None), ((1, 2, 3000, 128, 64), [1.0, 0.99]),
                                          ((1, 2, 300, 64, 128), [0.5, 0.9])],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else None)
def test_bwd_phi_tensor_core_path(shape, gammas, opts):
    """phi = elu + 1 without the normaliser: the three tensor-core passes over phi(q),
    phi(k) (reversed copies where a gamma is out of the reversed walk's range), the
    q and k gradients through phi' at the end, against the oracle."""
    opts.path("auto")
    B, H, T, dk, dv = shape
    seed = zlib.crc32(repr((shape, gammas, "bwd-phi")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16", gamma=gammas, phi=True)
    rng = np.random.default_rng(seed)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    S0 = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.3)
    dST = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.1)
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    la.trace_enable(4096)
    try:
        la.trace_collect()
        dq, dk_, dv_, dS0, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], phi=True, S0=S0.to(DEV),
                                            dS_T=dST.to(DEV))
        torch.cuda.synchronize()
        names = [n for n, _ in la.trace_collect()]
    finally:
        la.trace_enable(0)
    assert "phi_prep_kernel" in names and "phi_grad_pair_kernel" in names, names
    assert not any(n.startswith("chunk_bwd_simt") for n in names), names
    rq, rk, rv, rS0, _ = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO, phi=True,
                                              S0=S0, dS_T=dST)
    check("dq", to_np(dq), rq, TOL["bf16"])
    check("dk", to_np(dk_), rk, TOL["bf16"])
    check("dv", to_np(dv_), rv, TOL["bf16"])
    check("dS0", to_np(dS0), rS0, TOL["bf16"])


REVERSE_CASES = [  # shape, gammas, whether the kernel walks reversed time itself
    ((1, 2, 300, 64, 64), [1.0, 0.9], True),        # gamma = 1 beside gamma < 1; ragged tail
    ((2, 2, 3000, 64, 128), [0.999, 0.8], True),    # segments (scan), d_k != d_v
    ((2, 16, 1000, 128, 64), 0.97, True),           # segments folded in the output walk
    ((1, 1, 129, 128, 128), [0.71], True),         # near the factored form's floor: 0.71^127 = 2^-62.7
    ((1, 1, 1, 64, 64), [0.9], True),               # one token: the chunk starts 127 rows before 0
    ((2, 3, 100, 128, 64), [0.95, 1.0, 0.8], True),   # one partial chunk per sequence
    ((8, 16, 256, 64, 128), 0.99, True),             # more units than SMs: no segments
    ((1, 2, 300, 64, 64), [0.5, 0.9], False),       # gamma^127 < 2^-64: reversed copies
    ((1, 2, 3000, 128, 64), [0.6, 0.99], False),    # the same with segments
]


@pytest.mark.parametrize("shape,gammas,walk", REVERSE_CASES,
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else None)
def test_bwd_tensor_core_reversed_time(shape, gammas, walk, opts):
    """dK and dV come from forward passes in reversed time: by the pipelined kernel's
    own backward walk (chunks from the end, mirrored rows, the last chunk starting
    before row 0) where every gamma is in the factored form's range, else over
    reversed copies.  Both against the oracle, with an initial state and a
    final-state gradient; the trace shows which ran.  With segments, the dK pass
    takes the dV pass's segment contributions transposed (keys dO and values Q give
    the transpose of keys Q and values dO)."""
    opts.path("auto")
    B, H, T, dk, dv = shape
    seed = zlib.crc32(repr((shape, gammas, "bwd-rev")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16", gamma=gammas)
    rng = np.random.default_rng(seed)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    S0 = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.3)
    dST = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.1)
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    la.trace_enable(4096)
    try:
        la.trace_collect()
        dq, dk_, dv_, dS0, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], S0=S0.to(DEV),
                                            dS_T=dST.to(DEV))
        torch.cuda.synchronize()
        names = [n for n, _ in la.trace_collect()]
    finally:
        la.trace_enable(0)
    assert any(n.startswith("chunk_tc_ws_kernel") for n in names), names
    assert ("reverse_time_kernel" in names) == (not walk), names
    # segmented passes: the reversed walk runs the state walk of the dV pass only
    # and hands its transpose to the dK pass (two state walks, not three)
    assert names.count("chunk_tc_ws_kernel/state") in ((0, 2) if walk else (0, 3)), names
    rq, rk, rv, rS0, _ = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO, S0=S0,
                                              dS_T=dST)
    check("dq", to_np(dq), rq, TOL["bf16"])
    check("dk", to_np(dk_), rk, TOL["bf16"])
    check("dv", to_np(dv_), rv, TOL["bf16"])
    check("dS0", to_np(dS0), rS0, TOL["bf16"])


@pytest.mark.parametrize("gammas", [None, [0.5, 0.6]], ids=["walk", "copies"])
def test_bwd_tensor_core_path_repeated(gammas, opts):
    """The tensor-core composite twelve times over, its dV pass reading inputs written
    or read just before it (hot in L2): the case that once exposed an exit state read
    before the state walk's last MMA; both with the kernel's reversed walk and with
    reversed copies."""
    opts.path("auto")
    B, H, T, dk, dv = 1, 2, 3000, 64, 64
    x = workloads.random_case(9090, B, H, T, dk, dv, dtype="bf16", gamma=gammas)
    rng = np.random.default_rng(9090)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    rq, rk, rv, _, _ = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO)
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    for rep in range(12):
        dq, dk_, dv_, _, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], state_grads=False)
        torch.cuda.synchronize()
        check(f"dq (repeat {rep})", to_np(dq), rq, TOL["bf16"])
        check(f"dk (repeat {rep})", to_np(dk_), rk, TOL["bf16"])
        check(f"dv (repeat {rep})", to_np(dv_), rv, TOL["bf16"])


def test_bwd_matches_autograd_of_the_forward_kernel_inputs_on_fp32():
    """An fp32 case checked against torch autograd through the masked parallel form
    (an independent route to the same gradients, on the host)."""
    B, H, T, dk, dv = 1, 2, 40, 16, 16
    x = workloads.random_case(3, B, H, T, dk, dv, dtype="f32")
    q, k, v = (x[n].double().requires_grad_(True) for n in ("q", "k", "v"))
    g = torch.tensor(np.asarray(x["gamma"], np.float64))
    n = torch.arange(T, dtype=torch.float64)
    diff = n[:, None] - n[None, :]
    D = torch.where(diff >= 0, g[:, None, None] ** diff.clamp(min=0), torch.zeros(()))
    O = ((q @ k.transpose(-1, -2)) * D) @ v
    dO = torch.randn(B, H, T, dv, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    (O * dO).sum().backward()
    gq, gk, gv, _, _ = la.chunk_bwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV),
                                     dO.float().to(DEV), x["gamma"])
    torch.cuda.synchronize()
    check("dq", to_np(gq), q.grad.numpy(), TOL["f32"])
    check("dk", to_np(gk), k.grad.numpy(), TOL["f32"])
    check("dv", to_np(gv), v.grad.numpy(), TOL["f32"])


def test_bwd_linear_attention_bf16_full():
    """The linear-attention workload's shape (B4 H8 T4096 d64, phi, normalised; dk and
    dv on the tensor cores), every sequence's gradients against the oracle."""
    c = workloads.CONFIGS["linear_attention_bf16"]
    x = workloads.make_inputs(c)
    B, H, T, dv = c["B"], c["H"], c["T"], c["dv"]
    rng = np.random.default_rng(77)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    q, k, v, g_o = (t.to(DEV) for t in (x["q"], x["k"], x["v"], dO))
    dq, dk, dv_, _, _ = la.chunk_bwd(q, k, v, g_o, x["gamma"], phi=True, normalize=True)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO, phi=True,
                                            normalize=True)
    check("dq", to_np(dq), rq, TOL["bf16"])
    check("dk", to_np(dk), rk, TOL["bf16"])
    check("dv", to_np(dv_), rv, TOL["bf16"])


NORM_CASES = [  # shape, phi, floor, gammas, dk and dv on the tensor cores expected
    ((2, 2, 260, 64, 64), True, False, None, True),
    ((1, 3, 300, 128, 64), True, True, [1.0, 0.9, 0.8], True),
    ((1, 2, 300, 64, 64), False, True, [0.97, 0.99], True),
    ((2, 16, 1000, 64, 64), True, False, 1.0, True),       # segments folded in the walks
    ((1, 2, 3000, 64, 64), True, False, [1.0, 0.999], True),  # segments with a scan
    ((1, 1, 1, 64, 64), True, False, 0.9, True),             # one token
    ((3, 5, 129, 128, 64), True, True, None, True),          # a chunk and one row, d_k = 128
    ((1, 2, 200, 64, 64), True, False, [0.5, 0.9], False),   # gamma^127 < 2^-64: CUDA cores
    ((1, 2, 130, 64, 128), True, False, None, False),        # d_v = 128: CUDA cores
]


@pytest.mark.parametrize("shape,phi,floor,gammas,composite", NORM_CASES,
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else None)
def test_bwd_normalised_paths(shape, phi, floor, gammas, composite, opts):
    """The normalised backward: dq and the per-token dd, du from the CUDA-core kernel's
    forward sweep, then dk and dv as reversed-time tensor-core passes over [dn | du] and
    [v | 1] where they apply, the CUDA-core kernel's backward sweep otherwise; which ran
    is read from the launch trace.  With an initial state and final-state gradients,
    and dS_0, dz_0 checked too."""
    opts.path("auto")
    B, H, T, dk, dv = shape
    seed = zlib.crc32(repr((shape, phi, floor, gammas, "bwd-norm")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16", gamma=gammas, phi=phi,
                              normalize=True)
    rng = np.random.default_rng(seed)
    dO = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(torch.bfloat16)
    S0 = torch.from_numpy(np.abs(rng.standard_normal((B, H, dk, dv))).astype(np.float32) * 0.3)
    z0 = torch.from_numpy(np.abs(rng.standard_normal((B, H, dk))).astype(np.float32) + 0.5)
    dST = torch.from_numpy(rng.standard_normal((B, H, dk, dv)).astype(np.float32) * 0.1)
    dzT = torch.from_numpy(rng.standard_normal((B, H, dk)).astype(np.float32) * 0.1)
    q, k, v, g_o = (t.to(DEV).contiguous() for t in (x["q"], x["k"], x["v"], dO))
    la.trace_enable(4096)
    try:
        la.trace_collect()
        dq, dk_, dv_, dS0, dz0 = la.chunk_bwd(q, k, v, g_o, x["gamma"], phi=phi, normalize=True,
                                              floor=floor, S0=S0.to(DEV), z0=z0.to(DEV),
                                              dS_T=dST.to(DEV), dz_T=dzT.to(DEV))
        torch.cuda.synchronize()
        names = [n for n, _ in la.trace_collect()]
    finally:
        la.trace_enable(0)
    assert ("aug_prep_kernel" in names) == composite, names
    assert "chunk_bwd_simt_kernel/dq" in names, names
    assert ("chunk_bwd_simt_kernel/dkdv" in names) == (not composite), names
    rq, rk, rv, rS0, rz0 = oracle.recurrent_bwd(x["q"], x["k"], x["v"], x["gamma"], dO, phi=phi,
                                                normalize=True, floor=floor, S0=S0, z0=z0,
                                                dS_T=dST, dz_T=dzT)
    check("dq", to_np(dq), rq, TOL["bf16"])
    check("dk", to_np(dk_), rk, TOL["bf16"])
    check("dv", to_np(dv_), rv, TOL["bf16"])
    check("dS0", to_np(dS0), rS0, TOL["bf16"])
    check("dz0", to_np(dz0), rz0, TOL["bf16"])
