"""la_chunk_fwd_noalloc against la_chunk_fwd (GPU).

la_chunk_fwd_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns every device allocation, a serving loop that
must not allocate once running): it uses a fixed scratch array compiled into
the library instead of a caller workspace.  This file is named to be collected
last, so a run that stops at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import pins
import workloads

la = pytest.importorskip("retnet_retention_gb300")

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 tolerance of the parity tests
DEV = "cuda"
MAX_SCRATCH = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


def _case(seed):
    # few sequences, many chunks: the long-sequence split that needs scratch
    return workloads.random_case(seed, 1, 2, 4096, 64, 64, dtype="bf16")


def _with_workspace(x):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    O, S, z = la.chunk_fwd(q, k, v, x["gamma"], phi=True, normalize=True,
                           z_out=torch.empty(1, 2, 64, device=DEV))
    torch.cuda.synchronize()
    return O, S, z


def _no_alloc(x):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out = torch.empty_like(v)
    S = torch.empty(1, 2, 64, 64, device=DEV)
    z = torch.empty(1, 2, 64, device=DEV)
    la.chunk_fwd_noalloc(q, k, v, x["gamma"], phi=True, normalize=True, out=out, S_out=S,
                         z_out=z)
    torch.cuda.synchronize()
    return out, S, z


def _close(a, b, name):
    err = pins.rel_err(a.double().cpu().numpy(), b.double().cpu().numpy())
    assert err <= TOL, f"{name}: {err:.3e}"


def test_no_alloc_matches_workspace_entry_point_twice():
    assert la.workspace_size(1, 2, 4096, 64, 64, phi=True, normalize=True) > 0, \
        "this case must use scratch"
    for seed in (101, 202):  # two calls in a row, different inputs
        x = _case(seed)
        ref = _with_workspace(x)
        got = _no_alloc(x)
        for a, b, n in zip(got, ref, ("O", "S_T", "z_T")):
            _close(a, b, n)


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
