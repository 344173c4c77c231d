"""The tensor-core (tcgen05) chunkwise path against the fp64 oracle.

la_debug_set(LA_OPT_PATH, 2) pins la_chunk_fwd to the tensor-core kernels (an
error if the shape is outside them), la_debug_set(LA_OPT_PATH, 1) to the fp32
CUDA-core kernel;
both are compared with the oracle on the same seeded inputs, and with each
other.  Shapes cover one and several chunks of 128, ragged tails, T = 1,
d_k != d_v, both value-column block widths, the split of a long sequence into
segments (few sequences, many chunks), phi/normaliser, and the non-causal form.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


@pytest.fixture
def tc_path(opts):
    opts.path("tc")


@pytest.fixture(params=["pipelined", "lockstep"])
def tc_kernel(request, opts):
    """Both tensor-core output kernels: the warp-specialised pipeline (default
    where it applies) and the lockstep kernel (LA_OPT_TC_LOCKSTEP)."""
    opts.path("tc")
    if request.param == "lockstep":
        opts.lockstep(True)
    else:
        opts.lockstep(False)
    return request.param


def run(x, phi, normalize, causal=True, S0=None, z0=None, dev_status=None):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    B, H, T, dk = q.shape
    O, S, z = la.chunk_fwd(q, k, v, x["gamma"], phi=phi, normalize=normalize, causal=causal,
                           S0=S0, z0=z0, z_out=torch.empty(B, H, dk, device=DEV),
                           dev_status=dev_status)
    torch.cuda.synchronize()
    return (O.double().cpu().numpy(), S.double().cpu().numpy(), z.double().cpu().numpy())


def check(name, got, want, tol=TOL):
    assert np.all(np.isfinite(got)), f"{name}: non-finite"
    err = pins.rel_err(got, want)
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.0e}"


TC_SHAPES = [  # B, H, T, dk, dv
    (1, 2, 1, 64, 64),
    (2, 2, 128, 64, 64),
    (1, 3, 300, 128, 128),
    (2, 1, 129, 128, 256),
    (1, 2, 517, 64, 128),
    (1, 1, 384, 128, 64),
    (1, 2, 4100, 128, 128),   # few sequences, many chunks: segmented
    (1, 1, 2000, 64, 64),     # segmented with a ragged last segment
    (2, 16, 1000, 64, 64),    # 4 segments per sequence: entry states folded in the output walk
    (1, 40, 700, 128, 128),   # 3 segments per sequence, d_k = 128
]


@pytest.mark.parametrize("flags", [(False, False), (True, True), (True, False)],
                         ids=lambda f: f"phi{int(f[0])}_norm{int(f[1])}")
@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tc_matches_oracle(shape, flags, tc_kernel):
    B, H, T, dk, dv = shape
    phi, normalize = flags
    seed = zlib.crc32(repr((shape, flags, "tc")).encode()) % 100000
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16")
    O, S, z = run(x, phi, normalize)
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=phi,
                                  normalize=normalize)
    check("O", O, Or)
    check("S_T", S, Sr)
    check("z_T", z, zr)


@pytest.mark.parametrize("gamma", [[0.5, 0.9], [1.0, 0.999], [0.05, 0.99]])
def test_tc_decay_extremes(gamma, tc_kernel):
    """Small decays underflow instead of overflowing; gamma = 1 skips the scaling."""
    x = workloads.random_case(31, 1, 2, 700, 128, 128, dtype="bf16", gamma=gamma)
    O, S, _ = run(x, False, False)
    Or, Sr, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"])
    check("O", O, Or)
    check("S_T", S, Sr)


def test_tc_resume_from_state(tc_kernel):
    x = workloads.random_case(41, 2, 2, 900, 128, 128, dtype="bf16")
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True)
    t1 = 389
    a = {n: x[n][:, :, :t1].contiguous() for n in ("q", "k", "v")}
    b = {n: x[n][:, :, t1:].contiguous() for n in ("q", "k", "v")}
    a["gamma"] = b["gamma"] = x["gamma"]
    O1, S1, z1 = run(a, True, True)
    O2, S2, z2 = run(b, True, True, S0=torch.from_numpy(S1).float().to(DEV),
                     z0=torch.from_numpy(z1).float().to(DEV))
    check("O", np.concatenate([O1, O2], axis=2), Or)
    check("S_T", S2, Sr)
    check("z_T", z2, zr)


def test_tc_resume_from_state_folded_segments(tc_kernel):
    """A continued prefill whose entry states are folded from the segments'
    contributions and a nonzero initial state (32 sequences: 2-4 segments each)."""
    x = workloads.random_case(43, 2, 16, 1000, 64, 64, dtype="bf16")
    Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True)
    t1 = 389
    a = {n: x[n][:, :, :t1].contiguous() for n in ("q", "k", "v")}
    b = {n: x[n][:, :, t1:].contiguous() for n in ("q", "k", "v")}
    a["gamma"] = b["gamma"] = x["gamma"]
    O1, S1, z1 = run(a, True, True)
    O2, S2, z2 = run(b, True, True, S0=torch.from_numpy(S1).float().to(DEV),
                     z0=torch.from_numpy(z1).float().to(DEV))
    check("O", np.concatenate([O1, O2], axis=2), Or)
    check("S_T", S2, Sr)
    check("z_T", z2, zr)


def test_launch_count_follows_the_segment_plan():
    lib = la.library()
    assert lib.la_chunk_fwd_launches(2, 16, 1000, 64, 64, 1, 3, 0) == 2   # folded entry states
    assert lib.la_chunk_fwd_launches(1, 8, 65536, 128, 128, 1, 0, 0) == 3  # segment scan
    assert lib.la_chunk_fwd_launches(8, 16, 8192, 128, 256, 1, 0, 0) == 1  # one wave of units


@pytest.mark.parametrize("flags", [(False, False), (True, True)],
                         ids=lambda f: f"phi{int(f[0])}_norm{int(f[1])}")
def test_tc_noncausal(flags, tc_path):
    phi, normalize = flags
    x = workloads.random_case(51, 1, 3, 333, 128, 128, dtype="bf16", gamma=1.0)
    O, S, _ = run(x, phi, normalize, causal=False)
    Or, Sr, _ = oracle.noncausal(x["q"], x["k"], x["v"], phi=phi, normalize=normalize)
    check("O", O, Or)
    check("S", S, Sr)


def test_tc_and_simt_agree(opts):
    x = workloads.random_case(61, 2, 4, 640, 64, 64, dtype="bf16")
    opts.path("tc")
    Ot, St, zt = run(x, True, True)
    opts.path("simt")
    Os, Ss, zs = run(x, True, True)
    check("O", Ot, Os)
    check("S", St, Ss)
    check("z", zt, zs)


def test_tc_is_the_default_for_supported_shapes():
    assert la.library().la_chunk_fwd_launches(4, 8, 4096, 64, 64, 1, 3, 0) in (1, 2, 3)
    assert la.workspace_size(1, 8, 65536, 128, 128) > 0  # long and few: segmented


def test_timeout_is_reported_not_hung(opts, tc_kernel):
    """A wait that runs out (on a barrier nothing arrives on) sets dev_status; the
    context stays usable."""
    opts.force_timeout(True)
    x = workloads.random_case(71, 1, 2, 256, 64, 64, dtype="bf16")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run(x, False, False, dev_status=status)
    assert int(status.item()) == la.LA_ERR_TIMEOUT
    opts.force_timeout(False)
    status.zero_()
    O, S, _ = run(x, False, False, dev_status=status)
    assert int(status.item()) == 0
    Or, Sr, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"])
    check("O after a reported timeout", O, Or)


def test_launch_trace_names_the_kernels():
    x = workloads.random_case(81, 1, 1, 4096, 64, 64, dtype="bf16")
    la.trace_enable(64)
    try:
        run(x, True, True)
        recs = la.trace_collect()
    finally:
        la.trace_enable(0)
    names = [n for n, _ in recs]
    assert any(n.endswith("/full") for n in names), names
    assert all(ms > 0.0 for _, ms in recs)
    n = la.library().la_chunk_fwd_launches(1, 1, 4096, 64, 64, 1, 3, 0)
    assert len(names) == n, (names, n)
