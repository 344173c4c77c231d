"""la_chunk_fwd_noalloc against la_chunk_fwd and the fp64 oracle (GPU).

la_chunk_fwd_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns every device allocation, a serving loop that
must not allocate once running): it uses a fixed scratch array compiled into
the library instead of a caller workspace.  The cases cover a plan whose
segment contributions the output walk folds itself, a plan with the scan kernel
between the walks, and a call that needs no scratch at all.  This file is named
to be collected last, so a run that stops at the first failure has run every
other test first.
"""
import numpy as np
import pytest
import torch

import oracle
import pins
import workloads

la = pytest.importorskip("retnet_retention_gb300")

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 tolerance of the parity tests
DEV = "cuda"
MAX_SCRATCH = 16 << 20

# (B, H, T, d, phi and normaliser): few sequences, many chunks -> segments folded
# in the output walk; two long sequences without phi -> 76 segments and the scan
# kernel; two short chunks -> no segments and no scratch
CASES = [(1, 2, 4096, 64, True), (1, 2, 32768, 64, False), (1, 2, 200, 64, True)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


def _case(seed, B, H, T, d):
    return workloads.random_case(seed, B, H, T, d, d, dtype="bf16")


def _with_workspace(x, phi):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    B, H, _, d = q.shape
    O, S, z = la.chunk_fwd(q, k, v, x["gamma"], phi=phi, normalize=phi,
                           z_out=torch.empty(B, H, d, device=DEV))
    torch.cuda.synchronize()
    return O, S, z


def _no_alloc(x, phi):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    B, H, _, d = q.shape
    out = torch.empty_like(v)
    S = torch.empty(B, H, d, d, device=DEV)
    z = torch.empty(B, H, d, device=DEV)
    la.chunk_fwd_noalloc(q, k, v, x["gamma"], phi=phi, normalize=phi, out=out, S_out=S, z_out=z)
    torch.cuda.synchronize()
    return out, S, z


def _close(a, b, name):
    b = b if isinstance(b, np.ndarray) else b.double().cpu().numpy()
    err = pins.rel_err(a.double().cpu().numpy(), b)
    assert err <= TOL, f"{name}: {err:.3e}"


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_no_alloc_matches_workspace_entry_point_and_oracle_twice(case):
    B, H, T, d, phi = case
    need = la.workspace_size(B, H, T, d, d, phi=phi, normalize=phi)
    assert need <= MAX_SCRATCH
    if T > 1000:
        assert need > 0, "this case must use scratch"
    for seed in (101, 202):  # two calls in a row, different inputs
        x = _case(seed + T, B, H, T, d)
        ref = _with_workspace(x, phi)
        got = _no_alloc(x, phi)
        Or, Sr, zr = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=phi, normalize=phi)
        for a, b, want, n in zip(got, ref, (Or, Sr, zr), ("O", "S_T", "z_T")):
            _close(a, b, n + " against la_chunk_fwd")
            _close(a, want, n + " against the oracle")


def test_no_alloc_rejects_plans_beyond_its_scratch():
    # the long-sequence workload's segment plan needs more than the fixed array
    need = la.workspace_size(1, 8, 65536, 128, 128)
    if need <= MAX_SCRATCH:
        pytest.skip("this device's segment plan fits the fixed scratch")
    q = torch.zeros(1, 8, 65536, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    S = torch.empty(1, 8, 128, 128, device=DEV)
    with pytest.raises(la.LinAttnError) as e:
        la.chunk_fwd_noalloc(q, q, q, [0.99] * 8, out=out, S_out=S)
    assert e.value.status == la.LA_ERR_INVALID_ARG
