"""la_chunk_fwd inside a captured CUDA graph (GPU).

A caller that runs the same small forward over and over can capture it once and
replay it: the launches then cost no host work (the bench reports the replayed
step time beside the eager one).  With its outputs and workspace given, a
la_chunk_fwd call allocates nothing and launches only on the caller's stream, so
it can be captured.  Each case here captures one call, replays the graph on new
inputs copied into the captured buffers, and checks the outputs bit for bit
against an eager call on the same inputs: the same kernels run either way.
Cases: segments folded in the output walk (phi and the normaliser), segments
through the scan kernel, the per-token decay's pick kernel, the Taylor map.
"""
import zlib

import pytest
import torch

import workloads

la = pytest.importorskip("retnet_retention_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [  # B, H, T, dk, dv, phi, normalize, gated
    (4, 8, 2048, 64, 64, True, True, False),        # phi, normaliser, folded segments
    (1, 2, 20000, 128, 128, False, False, False),    # plain retention, scan kernel
    (2, 16, 1000, 128, 128, False, False, True),     # per-token decay, pick kernel
    (2, 4, 640, 16, 64, "taylor", True, False),      # Taylor features
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from retnet_retention_gb300 import _build
    _build.build()
    la.library()


def _inputs(seed, B, H, T, dk, dv, gated):
    x = workloads.random_case(seed, B, H, T, dk, dv, dtype="bf16", gate=gated)
    return {n: x[n].to(DEV).contiguous() for n in ("q", "k", "v")}, x


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_captured_forward_replays_like_an_eager_call(case):
    B, H, T, dk, dv, phi, normalize, gated = case
    seed = zlib.crc32(repr(case).encode()) % 100000
    dev_in, x = _inputs(seed, B, H, T, dk, dv, gated)
    ds = la.state_rows(dk, phi)
    gamma = None if gated else x["gamma"]
    log_a = x["log_a"].to(DEV).contiguous() if gated else None
    O = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=DEV)
    S = torch.empty(B, H, ds, dv, device=DEV)
    z = torch.empty(B, H, ds, device=DEV) if normalize else None
    need = la.workspace_size(B, H, T, dk, dv, torch.bfloat16, phi, normalize, gated=gated)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()

    def call(q, k, v, la_, out, s_out, z_out, stream):
        la.chunk_fwd(q, k, v, gamma, phi=phi, normalize=normalize, out=out, S_out=s_out,
                     z_out=z_out, workspace=ws, stream=stream, log_a=la_)

    # capture on buffers that the replay reads, after one eager call on the side stream
    q_c, k_c, v_c = (torch.zeros_like(dev_in[n]) for n in ("q", "k", "v"))
    la_c = torch.zeros_like(log_a) if gated else None
    with torch.cuda.stream(side):
        call(q_c, k_c, v_c, la_c, O, S, z, side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call(q_c, k_c, v_c, la_c, O, S, z, side)
    torch.cuda.synchronize()
    # new inputs into the captured buffers, then replay
    q_c.copy_(dev_in["q"]); k_c.copy_(dev_in["k"]); v_c.copy_(dev_in["v"])
    if gated:
        la_c.copy_(log_a)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        g.replay()
    torch.cuda.synchronize()
    # the eager call on the same inputs
    O_e = torch.empty_like(O)
    S_e = torch.empty_like(S)
    z_e = torch.empty_like(z) if normalize else None
    call(dev_in["q"], dev_in["k"], dev_in["v"], log_a, O_e, S_e, z_e, None)
    torch.cuda.synchronize()
    assert torch.isfinite(O.float()).all()
    assert torch.equal(O, O_e)
    assert torch.equal(S, S_e)
    if normalize:
        assert torch.equal(z, z_e)
