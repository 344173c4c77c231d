"""The C ABI on the host: the library loads, exports what include/linattn.h
declares, and rejects bad arguments before launching anything.

These tests make no compute call: every call below fails its host-side
checks (or is a pure size query), so they run without a GPU.  Device
pointers are fake, aligned or misaligned integers that are never touched.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import retnet_retention_gb300 as la

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")

FAKE = 0x10000000  # an aligned address that is never dereferenced
GAM = np.full(8, 0.9, dtype=np.float32)


@pytest.fixture(scope="module")
def lib():
    from retnet_retention_gb300 import _build
    _build.build()
    return la.library()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"LA_API\s+[\w\s\*]+?\b(la_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_symbols()
    assert set(names) >= {"la_state_init", "la_chunk_fwd", "la_recurrent_step",
                          "la_workspace_size", "la_status_string", "la_abi_version"}


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in linattn.h but not exported"


def test_binding_constants_match_the_header():
    """Every flag, status and dtype value the Python binding passes equals the
    header's definition (a drift would silently select another operation)."""
    text = open(HEADER).read()
    defined = {m[0]: int(m[1]) for m in re.findall(r"#define\s+(LA_[A-Z0-9_]+)\s+(\d+)u?\b", text)}
    defined.update({m[0]: int(m[1]) for m in re.findall(r"\b(LA_[A-Z0-9_]+)\s*=\s*(\d+)", text)})
    names = ["LA_OK", "LA_ERR_INVALID_ARG", "LA_ERR_UNSUPPORTED", "LA_ERR_CUDA", "LA_ERR_TIMEOUT",
             "LA_DTYPE_F32", "LA_DTYPE_BF16", "LA_PHI_ELU1", "LA_NORMALIZE", "LA_NONCAUSAL",
             "LA_NORM_FLOOR", "LA_GATED", "LA_PHI_TAYLOR", "LA_OPT_PATH", "LA_OPT_TC_LOCKSTEP",
             "LA_OPT_FORCE_TIMEOUT"]
    for name in names:
        assert getattr(la, name) == defined[name], name
    assert la.abi_version() == defined["LA_ABI_VERSION"]


def test_status_strings_and_version(lib):
    assert la.abi_version() == 1
    for code in range(5):
        assert la.status_string(code)
    assert la.status_string(77) == "unknown status"


def test_debug_switches_default_off_and_check_their_range(lib):
    """la_debug_set: every switch starts at 0, returns its previous value, and
    refuses unknown options and out-of-range values without changing anything."""
    for opt, hi in ((la.LA_OPT_PATH, 2), (la.LA_OPT_TC_LOCKSTEP, 1), (la.LA_OPT_FORCE_TIMEOUT, 1)):
        assert lib.la_debug_set(opt, 0) == 0
        assert lib.la_debug_set(opt, hi + 1) == -1
        assert lib.la_debug_set(opt, -1) == -1
        assert lib.la_debug_set(opt, hi) == 0
        assert lib.la_debug_set(opt, 0) == hi
    for bad in (0, 4, -1, 99):
        assert lib.la_debug_set(bad, 0) == -1
    with la.debug_options(path="simt", lockstep=True):
        assert lib.la_debug_set(la.LA_OPT_PATH, 1) == 1
        assert lib.la_debug_set(la.LA_OPT_TC_LOCKSTEP, 1) == 1
    assert lib.la_debug_set(la.LA_OPT_PATH, 0) == 0
    assert lib.la_debug_set(la.LA_OPT_TC_LOCKSTEP, 0) == 0
    with pytest.raises(ValueError):
        la.debug_set(la.LA_OPT_PATH, 7)


def test_library_reads_no_environment():
    """The shipped library takes no switch from the environment: the test
    switches go through la_debug_set only."""
    csrc = os.path.join(ROOT, "retnet_retention_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "getenv" not in text, f


def test_host_entry_point_sizes_and_rejections(lib):
    """la_host_arena_size and la_chunk_fwd_host's host checks (nothing is enqueued
    when they fail; the pointers below are never touched)."""
    n2 = lib.la_host_arena_size(4, 8, 64, 64, 64, 1, 0, 0, 2)
    assert n2 > 0
    assert lib.la_host_arena_size(4, 8, 64, 64, 64, 1, 0, 0, 5) == 0  # pieces > B
    assert lib.la_host_arena_size(4, 8, 64, 64, 64, 1, 0, 0, 0) == 0
    assert lib.la_host_arena_size(4, 8, 64, 64, 64, 1, 0, 0, 1) > n2 > lib.la_host_arena_size(
        4, 8, 64, 64, 64, 1, 0, 0, 4)

    def call(**over):
        a = dict(Q=FAKE, K=FAKE, V=FAKE, gamma=GAM.ctypes.data, O=FAKE, pieces=2, arena=FAKE,
                 arena_bytes=n2)
        a.update(over)
        return lib.la_chunk_fwd_host(a["Q"], a["K"], a["V"], 1, a["gamma"], 4, 8, 64, 64, 64, 0,
                                     1e-6, None, None, a["O"], None, None, 0, a["pieces"],
                                     a["arena"], a["arena_bytes"], None, None)

    for over in (dict(pieces=5), dict(pieces=0), dict(Q=None), dict(O=None), dict(gamma=None),
                 dict(arena_bytes=n2 - 1), dict(arena=FAKE + 8), dict(arena=None)):
        assert call(**over) == la.LA_ERR_INVALID_ARG, over
    bad = np.full(8, 1.5, dtype=np.float32)
    assert call(gamma=bad.ctypes.data) == la.LA_ERR_INVALID_ARG


def chunk(lib, **over):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, dtype=1, gamma=GAM.ctypes.data, B=2,
             H=8, T=64, dk=64, dv=64, flags=0, eps=1e-6, S0=None, z0=None, O=FAKE + 0x400000,
             S_out=None, z_out=None, chunk=0, ws=None, ws_bytes=0, st=None, stream=None)
    a.update(over)
    return lib.la_chunk_fwd(a["Q"], a["K"], a["V"], a["dtype"], a["gamma"], a["B"], a["H"],
                            a["T"], a["dk"], a["dv"], a["flags"], a["eps"], a["S0"], a["z0"],
                            a["O"], a["S_out"], a["z_out"], a["chunk"], a["ws"], a["ws_bytes"],
                            a["st"], a["stream"])


BAD_CHUNK_ARGS = [
    dict(B=-1), dict(H=-2), dict(T=-1), dict(dk=0), dict(dk=8), dict(dk=24), dict(dk=272),
    dict(dv=300), dict(dv=17), dict(dtype=2), dict(flags=64), dict(chunk=48), dict(chunk=256),
    dict(flags=la.LA_GATED),  # the per-token decay's planning flag: not a la_chunk_fwd flag
    dict(eps=float("nan")), dict(eps=-1.0), dict(Q=None), dict(V=None), dict(O=None),
    dict(Q=FAKE + 8), dict(O=FAKE + 0x400004), dict(S0=FAKE + 0x800004),
    dict(O=FAKE + 0x100000),  # O overlaps K
    dict(H=300, gamma=np.full(300, 0.9, dtype=np.float32).ctypes.data),
]


@pytest.mark.parametrize("over", BAD_CHUNK_ARGS, ids=lambda d: ",".join(f"{k}" for k in d))
def test_chunk_fwd_rejects(lib, over):
    assert chunk(lib, **over) == la.LA_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [0.0, -0.5, 1.0001, float("nan"), float("inf")])
def test_chunk_fwd_rejects_gamma(lib, bad):
    g = GAM.copy()
    g[3] = bad
    assert chunk(lib, gamma=g.ctypes.data) == la.LA_ERR_INVALID_ARG


def test_noncausal_needs_gamma_one_and_no_state(lib):
    ones = np.ones(8, dtype=np.float32)
    assert chunk(lib, flags=la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED  # gamma 0.9
    assert chunk(lib, flags=la.LA_NONCAUSAL, gamma=ones.ctypes.data,
                 S0=FAKE + 0x800000) == la.LA_ERR_UNSUPPORTED


def test_empty_batch_is_a_noop(lib):
    # B == 0: nothing to do, no pointer is needed
    assert chunk(lib, B=0, Q=None, K=None, V=None, O=None, gamma=None) == la.LA_OK


def test_workspace_size_is_a_host_query(lib):
    for (B, H, T, dk, dv) in [(4, 8, 4096, 64, 64), (8, 16, 8192, 128, 256),
                              (1, 8, 65536, 128, 128), (0, 1, 1, 16, 16)]:
        n = lib.la_workspace_size(B, H, T, dk, dv, 1, 0, 0)
        assert n >= 0 and n % 16 == 0


def chunk_gated(lib, **over):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, dtype=1, log_a=FAKE + 0x300000, B=2,
             H=8, T=64, dk=64, dv=64, flags=0, eps=1e-6, S0=None, z0=None, O=FAKE + 0x400000,
             S_out=None, z_out=None, chunk=0, ws=None, ws_bytes=0, st=None, stream=None)
    a.update(over)
    return lib.la_chunk_fwd_gated(a["Q"], a["K"], a["V"], a["dtype"], a["log_a"], a["B"],
                                  a["H"], a["T"], a["dk"], a["dv"], a["flags"], a["eps"], a["S0"],
                                  a["z0"], a["O"], a["S_out"], a["z_out"], a["chunk"], a["ws"],
                                  a["ws_bytes"], a["st"], a["stream"])


@pytest.mark.parametrize("over", [dict(log_a=None), dict(log_a=FAKE + 0x300004), dict(B=-1),
                                  dict(dk=24), dict(flags=64), dict(Q=None), dict(eps=-1.0),
                                  dict(log_a=FAKE + 0x400000)],  # O overlaps log_a
                         ids=lambda d: ",".join(d))
def test_chunk_fwd_gated_rejects(lib, over):
    assert chunk_gated(lib, **over) == la.LA_ERR_INVALID_ARG


def test_chunk_fwd_gated_noncausal_unsupported_and_empty_batch(lib):
    assert chunk_gated(lib, flags=la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED
    assert chunk_gated(lib, B=0, Q=None, K=None, V=None, O=None, log_a=None) == la.LA_OK


def test_workspace_size_takes_the_gated_flag(lib):
    for (B, H, T, dk, dv) in [(4, 8, 4096, 64, 64), (1, 8, 65536, 128, 128)]:
        n = lib.la_workspace_size(B, H, T, dk, dv, 1, la.LA_GATED, 0)
        assert n >= 0 and n % 16 == 0
    assert lib.la_workspace_size(4, 8, 4096, 64, 64, 1, 64, 0) == 0  # unknown flag


def bwd(lib, gated=False, **over):
    a = dict(Q=FAKE, K=FAKE + 0x100000, V=FAKE + 0x200000, dO=FAKE + 0x300000, dtype=1,
             gamma=GAM.ctypes.data, log_a=FAKE + 0x900000, B=2, H=8, T=64, dk=64, dv=64, flags=0,
             eps=1e-6, S0=None, z0=None, dST=None, dzT=None, dQ=FAKE + 0x400000,
             dK=FAKE + 0x500000, dV=FAKE + 0x600000, dS0=None, dz0=None, ws=None, ws_bytes=0,
             st=None, stream=None)
    a.update(over)
    fn = lib.la_chunk_bwd_gated if gated else lib.la_chunk_bwd
    return fn(a["Q"], a["K"], a["V"], a["dO"], a["dtype"], a["log_a"] if gated else a["gamma"],
              a["B"], a["H"], a["T"], a["dk"], a["dv"], a["flags"], a["eps"], a["S0"], a["z0"],
              a["dST"], a["dzT"], a["dQ"], a["dK"], a["dV"], a["dS0"], a["dz0"], a["ws"],
              a["ws_bytes"], a["st"], a["stream"])


@pytest.mark.parametrize("over", [dict(B=-1), dict(dk=24), dict(dtype=3), dict(flags=64),
                                  dict(dO=None), dict(dQ=None), dict(dK=FAKE + 0x500008),
                                  dict(dQ=FAKE + 0x300000),   # dQ overlaps dO
                                  dict(dV=FAKE + 0x400000),   # dV overlaps dQ
                                  dict(flags=la.LA_NORMALIZE),  # no workspace for the denominators
                                  dict(eps=-1.0)],
                         ids=lambda d: ",".join(d))
def test_chunk_bwd_rejects(lib, over):
    assert bwd(lib, **over) == la.LA_ERR_INVALID_ARG


def test_chunk_bwd_unsupported_and_sizes(lib):
    assert bwd(lib, flags=la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED
    assert bwd(lib, dk=256) == la.LA_ERR_UNSUPPORTED
    assert bwd(lib, gated=True, log_a=None) == la.LA_ERR_INVALID_ARG
    assert bwd(lib, B=0, Q=None, K=None, V=None, dO=None, dQ=None, dK=None, dV=None) == la.LA_OK
    n = lib.la_bwd_workspace_size(2, 8, 64, 64, 64, 1, la.LA_NORMALIZE)
    assert n == 2 * 8 * 64 * 2 * 4
    assert lib.la_bwd_workspace_size(2, 8, 64, 64, 64, 1, 0) == 0
    assert lib.la_bwd_workspace_size(2, 8, 64, 256, 64, 1, 0) == 0  # unsupported


def step(lib, **over):
    a = dict(q=FAKE, k=FAKE + 0x1000, v=FAKE + 0x2000, dtype=1, gamma=GAM.ctypes.data, B=2, H=8,
             dk=64, dv=64, flags=0, eps=1e-6, S=FAKE + 0x100000, z=None, o=FAKE + 0x200000,
             st=None, stream=None)
    a.update(over)
    return lib.la_recurrent_step(a["q"], a["k"], a["v"], a["dtype"], a["gamma"], a["B"], a["H"],
                                 a["dk"], a["dv"], a["flags"], a["eps"], a["S"], a["z"], a["o"],
                                 a["st"], a["stream"])


@pytest.mark.parametrize("over", [dict(B=-1), dict(dk=20), dict(dv=512), dict(S=None),
                                  dict(o=None), dict(flags=la.LA_NORMALIZE), dict(flags=la.LA_NORM_FLOOR),  # z missing
                                  dict(q=FAKE + 2), dict(S=FAKE + 0x100008), dict(dtype=5),
                                  dict(o=FAKE + 0x100000)],  # o overlaps S
                         ids=lambda d: ",".join(d))
def test_recurrent_step_rejects(lib, over):
    assert step(lib, **over) == la.LA_ERR_INVALID_ARG


def test_recurrent_step_noncausal_unsupported(lib):
    assert step(lib, flags=la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED


def test_recurrent_step_gated_rejects(lib):
    def call(log_a, flags=0):
        return lib.la_recurrent_step_gated(FAKE, FAKE + 0x1000, FAKE + 0x2000, 1, log_a, 2, 8, 64,
                                           64, flags, 1e-6, FAKE + 0x100000, None,
                                           FAKE + 0x200000, None, None)
    assert call(None) == la.LA_ERR_INVALID_ARG
    assert call(FAKE + 0x300004) == la.LA_ERR_INVALID_ARG
    assert call(FAKE + 0x300000, flags=la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED


def test_state_init_rejects(lib):
    assert lib.la_state_init(None, None, 2, 2, 64, 64, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_state_init(FAKE + 4, None, 2, 2, 64, 64, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_state_init(FAKE, None, 2, 2, 63, 64, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_state_init(None, None, 0, 2, 64, 64, None) == la.LA_OK


def test_python_binding_refuses_host_tensors():
    """Host tensors never reach the library (their addresses are not device memory)."""
    import torch
    q = torch.zeros(1, 1, 4, 16)
    with pytest.raises(ValueError):
        la.chunk_fwd(q, q, q, [0.5], out=q.clone(), return_state=False)
    with pytest.raises(ValueError):
        la.recurrent_step(q[:, :, 0], q[:, :, 0], q[:, :, 0], [0.5], torch.zeros(1, 1, 16, 16),
                          out=q[:, :, 0].clone())


TAYLOR_UNSUPPORTED = [
    dict(dk=64), dict(dk=32), dict(dtype=0), dict(dv=48), dict(dv=16), dict(chunk=64),
    dict(flags=la.LA_PHI_TAYLOR | la.LA_PHI_ELU1), dict(flags=la.LA_PHI_TAYLOR | la.LA_NONCAUSAL),
]


@pytest.mark.parametrize("over", TAYLOR_UNSUPPORTED, ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_taylor_outside_its_kernel_is_unsupported(lib, over):
    """The Taylor feature map runs for bf16, d_k = 16, d_v a multiple of 64, causal,
    without elu + 1 and with chunk 0 or 128; other combinations are refused before
    any launch."""
    a = dict(dk=16, dv=64, flags=la.LA_PHI_TAYLOR)
    a.update(over)
    assert chunk(lib, **a) == la.LA_ERR_UNSUPPORTED


def test_taylor_outside_the_decode_steps_and_the_backward_passs_shapes(lib):
    """The decode step and the backward pass take the Taylor map for 16-wide q and k,
    not with elu + 1 (and the backward not with per-token decays); the chunkwise
    forward with per-token decays not at all."""
    assert step(lib, dk=64, flags=la.LA_PHI_TAYLOR) == la.LA_ERR_UNSUPPORTED
    assert step(lib, dk=16, flags=la.LA_PHI_TAYLOR | la.LA_PHI_ELU1) == la.LA_ERR_UNSUPPORTED
    assert step(lib, dk=16, flags=la.LA_PHI_TAYLOR | la.LA_NONCAUSAL) == la.LA_ERR_UNSUPPORTED
    assert bwd(lib, dk=64, flags=la.LA_PHI_TAYLOR) == la.LA_ERR_UNSUPPORTED
    assert bwd(lib, dk=16, flags=la.LA_PHI_TAYLOR | la.LA_PHI_ELU1) == la.LA_ERR_UNSUPPORTED
    assert chunk_gated(lib, dk=16, flags=la.LA_PHI_TAYLOR) == la.LA_ERR_UNSUPPORTED
    assert lib.la_bwd_workspace_size(2, 8, 64, 16, 64, 1, la.LA_PHI_TAYLOR | la.LA_GATED) == 0
    assert lib.la_bwd_workspace_size(2, 8, 64, 64, 64, 1, la.LA_PHI_TAYLOR) == 0
    # the normalised call's workspace holds the per-token denominators at least
    assert lib.la_bwd_workspace_size(2, 8, 64, 16, 64, 1, la.LA_PHI_TAYLOR | la.LA_NORMALIZE) >= 2 * 8 * 64 * 8


def test_taylor_plan_queries(lib):
    """No workspace and one launch: the feature map's kernel has no segment plan."""
    f = la.LA_PHI_TAYLOR | la.LA_NORMALIZE
    assert lib.la_workspace_size(8, 16, 4096, 16, 64, 1, f, 0) == 0
    assert lib.la_chunk_fwd_launches(8, 16, 4096, 16, 64, 1, f, 0) == 1
    assert la.state_rows(16, "taylor") == 273 and la.state_rows(16) == 16
    with pytest.raises(ValueError):
        la._flags("softmax", False, True)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library the binding raises: no compute falls back to the host."""
    monkeypatch.setattr(la, "_LIB", None)
    monkeypatch.setattr(la, "LIBRARY_PATH", str(tmp_path / "liblinattn.so"))
    with pytest.raises(RuntimeError, match="not built"):
        la.library()
    import torch
    q = torch.zeros(1, 1, 4, 16)
    with pytest.raises((RuntimeError, ValueError)):
        la.chunk_fwd(q, q, q, [0.9])


def test_python_binding_checks_caller_buffers():
    """Caller-supplied outputs, states and gradients are checked for element count,
    dtype and device before their addresses reach the library (which cannot see a
    tensor's size): an undersized or mistyped buffer is refused, not written past."""
    import torch
    B, H, T, d = 2, 3, 8, 16
    q = torch.zeros(B, H, T, d, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out holds"):
        la.chunk_fwd(q, q, q, [0.5], out=torch.empty(B, H, T - 1, d, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="out must be"):
        la.chunk_fwd(q, q, q, [0.5], out=torch.empty(B, H, T, d))
    with pytest.raises(TypeError, match="S0 must be"):
        la.chunk_fwd(q, q, q, [0.5], S0=torch.zeros(B, H, d, d, dtype=torch.float64))
    with pytest.raises(ValueError, match="S0 holds"):  # the Taylor map's states have 273 rows
        la.chunk_fwd(q, q, torch.zeros(B, H, T, 64, dtype=torch.bfloat16), [0.5], phi="taylor",
                     S0=torch.zeros(B, H, d, 64))
    with pytest.raises(ValueError, match="z_out holds"):
        la.chunk_fwd(q, q, q, [0.5], normalize=True, z_out=torch.empty(B, H, d - 1))
    with pytest.raises(TypeError, match="dev_status must be"):
        la.chunk_fwd(q, q, q, [0.5], dev_status=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="S_out holds"):
        la.chunk_fwd_noalloc(q, q, q, [0.5], out=torch.empty_like(q), S_out=torch.empty(B, H, d))
    with pytest.raises(ValueError, match="shape mismatch"):
        la.chunk_fwd_noalloc(q, q[:, :, :4], q, [0.5], out=torch.empty_like(q),
                             S_out=torch.empty(B, H, d, d))
    s = q[:, :, 0].contiguous()
    with pytest.raises(ValueError, match="shape mismatch"):
        la.recurrent_step(s, s[:1], s, [0.5], torch.zeros(B, H, d, d))
    with pytest.raises(ValueError, match="S holds"):
        la.recurrent_step(s, s, s, [0.5], torch.zeros(B, H, d, d - 1))
    with pytest.raises(ValueError, match="z holds"):
        la.recurrent_step(s, s, s, [0.5], torch.zeros(B, H, d, d), torch.zeros(B, H, 1),
                          normalize=True)
    with pytest.raises(ValueError, match="dq holds"):
        la.chunk_bwd(q, q, q, q, [0.5], dq=torch.empty(B, H, T, d - 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="dS_T holds"):
        la.chunk_bwd(q, q, q, q, [0.5], dS_T=torch.zeros(B, H, d))
    with pytest.raises(ValueError, match="log_a must be"):
        la.chunk_bwd(q, q, q, q, log_a=torch.zeros(B, H, T - 1))
    with pytest.raises(ValueError, match="z holds"):
        la.state_init(torch.zeros(B, H, d, d), torch.zeros(B, H, d - 1))
    with pytest.raises(TypeError, match="S must be"):
        la.state_init(torch.zeros(B, H, d, d, dtype=torch.bfloat16))
    # buffers of the right size still fail only on being host memory
    with pytest.raises(ValueError, match="CUDA device tensors"):
        la.chunk_fwd(q, q, q, [0.5], out=torch.empty_like(q), S_out=torch.empty(B, H, d, d))
