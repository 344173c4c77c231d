"""Python binding of liblinattn.so: causal decayed linear attention on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels behind the C ABI (include/linattn.h); PyTorch supplies device memory
and the current stream.  There is no CPU fallback: without the built library
every call raises.

Names follow the C ABI:
  state_init(S, z=None)                        zero a state        (la_state_init)
  chunk_fwd(q, k, v, gamma, ...)               prefill / forward   (la_chunk_fwd)
  chunk_fwd(q, k, v, log_a=..., ...)           per-token decay     (la_chunk_fwd_gated)
  chunk_bwd(q, k, v, dO, gamma, ...)           gradients           (la_chunk_bwd[_gated])
  recurrent_step(q, k, v, gamma, S, z, ...)    one decode step     (la_recurrent_step)
  recurrent_step(q, k, v, None, S, z, log_a=)  per-token decay     (la_recurrent_step_gated)
  workspace_size(...)                          scratch bytes       (la_workspace_size)
  chunk_fwd_host(...)                          host buffers, copies included (la_chunk_fwd_host)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(5)
LA_DTYPE_F32, LA_DTYPE_BF16 = 0, 1
LA_PHI_ELU1, LA_NORMALIZE, LA_NONCAUSAL, LA_NORM_FLOOR, LA_GATED, LA_PHI_TAYLOR = 1, 2, 4, 8, 16, 32
LA_OPT_PATH, LA_OPT_TC_LOCKSTEP, LA_OPT_FORCE_TIMEOUT = 1, 2, 3

LIBRARY_PATH = _build.LIBRARY
_LIB = None


class TraceRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char_p), ("ms", ctypes.c_float)]


def trace_enable(capacity: int = 4096):
    """Record CUDA events around every library kernel launch (0 disables)."""
    _check(_load().la_trace_enable(int(capacity)), "la_trace_enable")


def trace_collect(max_records: int = 4096) -> list[tuple[str, float]]:
    """(kernel name, device ms) of every launch traced since the last collect."""
    buf = (TraceRecord * max_records)()
    n = _load().la_trace_collect(buf, max_records)
    if n < 0:
        raise LinAttnError(-n, "la_trace_collect")
    return [(buf[i].kernel.decode(), float(buf[i].ms)) for i in range(n)]


class LinAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIBRARY_PATH):
        raise RuntimeError(
            f"{LIBRARY_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`"
            " (or retnet_retention_gb300/_build.py) first")
    lib = ctypes.CDLL(LIBRARY_PATH)
    vp, i, u, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
    lib.la_status_string.argtypes = [i]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_abi_version.restype = i
    lib.la_workspace_size.argtypes = [i, i, i, i, i, i, u, i]
    lib.la_workspace_size.restype = sz
    lib.la_state_init.argtypes = [vp, vp, i, i, i, i, vp]
    lib.la_state_init.restype = i
    lib.la_chunk_fwd.argtypes = [vp, vp, vp, i, vp, i, i, i, i, i, u, f, vp, vp, vp, vp, vp, i,
                                 vp, sz, vp, vp]
    lib.la_chunk_fwd.restype = i
    lib.la_recurrent_step.argtypes = [vp, vp, vp, i, vp, i, i, i, i, u, f, vp, vp, vp, vp, vp]
    lib.la_recurrent_step.restype = i
    lib.la_chunk_fwd_gated.argtypes = lib.la_chunk_fwd.argtypes
    lib.la_chunk_fwd_gated.restype = i
    lib.la_recurrent_step_gated.argtypes = lib.la_recurrent_step.argtypes
    lib.la_recurrent_step_gated.restype = i
    lib.la_chunk_bwd.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, i, u, f, vp, vp, vp, vp,
                                 vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.la_chunk_bwd.restype = i
    lib.la_chunk_bwd_gated.argtypes = lib.la_chunk_bwd.argtypes
    lib.la_chunk_bwd_gated.restype = i
    lib.la_bwd_workspace_size.argtypes = [i, i, i, i, i, i, u]
    lib.la_bwd_workspace_size.restype = sz
    lib.la_chunk_fwd_launches.argtypes = [i, i, i, i, i, i, u, i]
    lib.la_chunk_fwd_launches.restype = i
    lib.la_chunk_fwd_noalloc.argtypes = [vp, vp, vp, i, vp, i, i, i, i, i, u, f, vp, vp, vp, vp,
                                         vp, i, vp, vp]
    lib.la_chunk_fwd_noalloc.restype = i
    lib.la_host_arena_size.argtypes = [i, i, i, i, i, i, u, i, i]
    lib.la_host_arena_size.restype = sz
    lib.la_chunk_fwd_host.argtypes = [vp, vp, vp, i, vp, i, i, i, i, i, u, f, vp, vp, vp, vp, vp,
                                      i, i, vp, sz, vp, vp]
    lib.la_chunk_fwd_host.restype = i
    lib.la_debug_set.argtypes = [i, i]
    lib.la_debug_set.restype = i
    lib.la_trace_enable.argtypes = [i]
    lib.la_trace_enable.restype = i
    lib.la_trace_collect.argtypes = [ctypes.POINTER(TraceRecord), i]
    lib.la_trace_collect.restype = i
    _LIB = lib
    return lib


def library() -> ctypes.CDLL:
    """The loaded liblinattn.so (raises if it is not built)."""
    return _load()


_PATHS = {"auto": 0, "simt": 1, "tc": 2}


def debug_set(option: int, value: int) -> int:
    """la_debug_set: set a test / diagnostic switch, return its previous value."""
    prev = int(_load().la_debug_set(int(option), int(value)))
    if prev < 0:
        raise ValueError(f"la_debug_set: bad option {option} or value {value}")
    return prev


class debug_options:
    """Context manager over la_debug_set's switches, restoring them on exit:
    path ("auto", "simt": CUDA cores, "tc": tensor cores), lockstep (the
    tensor-core forward's lockstep kernel), force_timeout (the kernels' forced
    1 ms wait and LA_ERR_TIMEOUT status)."""

    def __init__(self, path: str | None = None, lockstep: bool | None = None,
                 force_timeout: bool | None = None):
        self._set = []
        if path is not None:
            self._set.append((LA_OPT_PATH, _PATHS[path]))
        if lockstep is not None:
            self._set.append((LA_OPT_TC_LOCKSTEP, int(bool(lockstep))))
        if force_timeout is not None:
            self._set.append((LA_OPT_FORCE_TIMEOUT, int(bool(force_timeout))))
        self._prev = []

    def __enter__(self):
        self._prev = [(o, debug_set(o, v)) for o, v in self._set]
        return self

    def __exit__(self, *exc):
        for o, v in reversed(self._prev):
            debug_set(o, v)
        return False


def status_string(status: int) -> str:
    return _load().la_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_load().la_abi_version())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return LA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _flags(phi, normalize: bool, causal: bool, floor: bool = False) -> int:
    """phi: False (identity), True (elu + 1) or "taylor" (the second-order Taylor map)."""
    if phi == "taylor":
        fm = LA_PHI_TAYLOR
    elif phi is True or phi is False:
        fm = LA_PHI_ELU1 if phi else 0
    else:
        raise ValueError(f"phi must be False, True or 'taylor', not {phi!r}")
    return fm | (LA_NORMALIZE if normalize else 0) | (0 if causal else LA_NONCAUSAL) | (
        LA_NORM_FLOOR if floor else 0)


def state_rows(dk: int, phi=False) -> int:
    """Rows of the state S (and entries of z) for queries and keys of width dk:
    dk, or 1 + dk + dk^2 with the Taylor feature map."""
    return 1 + dk + dk * dk if phi == "taylor" else dk


def _ptr(t) -> int | None:
    """Device address of a contiguous CUDA tensor (None passes through)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("liblinattn takes CUDA device tensors (use chunk_fwd_host for host data)")
    if not t.is_contiguous():
        raise ValueError("tensors passed to liblinattn must be contiguous")
    return t.data_ptr()


def _buffer(t, name: str, numel: int, dtype, device):
    """Check a caller-supplied tensor before its address goes to the library, which
    reads or writes `numel` elements of `dtype` there and cannot see the tensor's
    size: a smaller, differently typed or misplaced tensor is refused (None passes)."""
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}; the inputs are on {device}")
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; {numel} are needed")


def _inputs(dev, **ts):
    """Every input tensor on the device of the first (the library sees addresses only)."""
    for name, t in ts.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}; the inputs are on {dev}")


def _workspace(ws, need: int, dev) -> int:
    """Check a caller-supplied workspace (uint8, contiguous, on dev, >= need bytes);
    returns its size in bytes."""
    if ws is None:
        return 0
    _buffer(ws, "workspace", need, torch.uint8, dev)
    if not ws.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return ws.numel()


def _states(B: int, H: int, ds: int, dv: int, device, **bufs):
    """The fp32 states and normalisers of a call: S-like [B,H,ds,dv], z-like [B,H,ds]."""
    for name, t in bufs.items():
        _buffer(t, name, B * H * ds * (1 if name.startswith(("z", "dz")) else dv),
                torch.float32, device)


def _gamma_host(gamma, H: int) -> np.ndarray:
    if isinstance(gamma, torch.Tensor):
        gamma = gamma.detach().to("cpu", torch.float32).numpy()
    g = np.ascontiguousarray(np.broadcast_to(np.asarray(gamma, dtype=np.float32).reshape(-1),
                                             (H,)), dtype=np.float32)
    return g


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _check(status: int, what: str):
    if status != LA_OK:
        raise LinAttnError(status, what)


def workspace_size(B, H, T, dk, dv, dtype=torch.bfloat16, phi=False, normalize=False,
                   causal=True, chunk=0, gated=False, floor=False) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    flags = _flags(phi, normalize, causal, floor) | (LA_GATED if gated else 0)
    return int(_load().la_workspace_size(B, H, T, dk, dv, code, flags, chunk))


def state_init(S: torch.Tensor, z: torch.Tensor | None = None, stream=None):
    """Zero S [B,H,dk,dv] (and z [B,H,dk]) on the device."""
    B, H, dk, dv = S.shape
    _states(B, H, dk, dv, S.device, S=S, z=z)
    _check(_load().la_state_init(_ptr(S), _ptr(z), B, H, dk, dv, _stream(stream)),
           "la_state_init")


def chunk_fwd(q, k, v, gamma=None, *, phi=False, normalize=False, causal=True, eps=1e-6,
              S0=None, z0=None, chunk=0, out=None, S_out=None, z_out=None, return_state=True,
              workspace=None, dev_status=None, stream=None, floor=False, log_a=None):
    """Chunkwise forward over [B,H,T,d] device tensors.

    Returns (O, S_T, z_T); S_T / z_T are None when return_state is False and
    no output buffer was given.  z_T is returned when normalising (or when
    z_out is given).  floor=True divides by max(|phi(q)^T z|, 1) (LA_NORM_FLOOR;
    implies normalising, eps unused).  log_a: a [B,H,T] fp32 device tensor of
    per-token log decays used instead of gamma (la_chunk_fwd_gated).
    phi="taylor": the second-order Taylor feature map (LA_PHI_TAYLOR; bf16,
    d = 16); the states then have state_rows(d, "taylor") = 273 rows.
    """
    normalize = normalize or floor
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    dt = _dtype_code(q)
    dev = q.device
    _inputs(dev, k=k, v=v)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=dev)
    ds = state_rows(dk, phi)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, ds, dv), dtype=torch.float32, device=dev)
    if return_state and normalize and z_out is None:
        z_out = torch.empty((B, H, ds), dtype=torch.float32, device=dev)
    if (gamma is None) == (log_a is None):
        raise ValueError("pass exactly one of gamma and log_a")
    if log_a is not None and (log_a.dtype != torch.float32 or tuple(log_a.shape) != (B, H, T)):
        raise ValueError(f"log_a must be float32 [B,H,T] = {(B, H, T)}")
    _buffer(log_a, "log_a", B * H * T, torch.float32, dev)
    _buffer(out, "out", B * H * T * dv, q.dtype, dev)
    _states(B, H, ds, dv, dev, S0=S0, z0=z0, S_out=S_out, z_out=z_out)
    _buffer(dev_status, "dev_status", 1, torch.int32, dev)
    flags = _flags(phi, normalize, causal, floor)
    lib = _load()
    with _current(dev):  # the plan (SM count) and the launches are the current device's
        need = int(lib.la_workspace_size(B, H, T, dk, dv, dt,
                                         flags | (LA_GATED if log_a is not None else 0), chunk))
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = _workspace(workspace, need, dev)
        if log_a is None:
            g = _gamma_host(gamma, H)
            st = lib.la_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), dt, g.ctypes.data, B, H, T, dk, dv,
                                  flags, float(eps), _ptr(S0), _ptr(z0), _ptr(out), _ptr(S_out),
                                  _ptr(z_out), int(chunk), _ptr(workspace), ws_bytes,
                                  _ptr(dev_status), _stream(stream))
            _check(st, "la_chunk_fwd")
        else:
            st = lib.la_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(log_a), B, H, T, dk,
                                        dv, flags, float(eps), _ptr(S0), _ptr(z0), _ptr(out),
                                        _ptr(S_out), _ptr(z_out), int(chunk), _ptr(workspace),
                                        ws_bytes, _ptr(dev_status), _stream(stream))
            _check(st, "la_chunk_fwd_gated")
    return out, S_out, z_out


def _current(dev):
    """The library plans and launches on the current device: make the tensors' current."""
    if dev.type != "cuda":
        raise ValueError("liblinattn takes CUDA device tensors (use chunk_fwd_host for host data)")
    return torch.cuda.device(dev)


def chunk_fwd_noalloc(q, k, v, gamma, *, phi=False, normalize=False, causal=True, eps=1e-6,
                      S0=None, z0=None, chunk=0, out=None, S_out=None, z_out=None,
                      dev_status=None, stream=None, floor=False):
    """chunk_fwd through la_chunk_fwd_noalloc: no workspace argument; the library's
    fixed scratch array is used instead (for callers that cannot allocate device
    memory).  out / S_out / z_out must be given: this call allocates nothing."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if out is None or S_out is None:
        raise ValueError("chunk_fwd_noalloc allocates nothing: pass out and S_out")
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    _inputs(q.device, k=k, v=v)
    _buffer(out, "out", B * H * T * dv, q.dtype, q.device)
    _states(B, H, state_rows(dk, phi), dv, q.device, S0=S0, z0=z0, S_out=S_out, z_out=z_out)
    _buffer(dev_status, "dev_status", 1, torch.int32, q.device)
    g = _gamma_host(gamma, H)
    with _current(q.device):  # the scratch array and the plan are the current device's
        st = _load().la_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), g.ctypes.data,
                                          B, H, T, dk, dv, _flags(phi, normalize, causal, floor),
                                          float(eps), _ptr(S0), _ptr(z0), _ptr(out), _ptr(S_out),
                                          _ptr(z_out), int(chunk), _ptr(dev_status),
                                          _stream(stream))
    _check(st, "la_chunk_fwd_noalloc")
    return out, S_out, z_out


def recurrent_step(q, k, v, gamma, S, z=None, *, phi=False, normalize=False, eps=1e-6,
                   out=None, dev_status=None, stream=None, floor=False, log_a=None):
    """One decode step on [B,H,d] device tensors; S (and z) are updated in place.
    floor=True: divide by max(|phi(q)^T z|, 1) (needs z).  log_a: this step's
    per-token log decays, a [B,H] fp32 device tensor, instead of gamma."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:2] != q.shape[:2]:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    _inputs(q.device, k=k, v=v)
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    if (gamma is None) == (log_a is None):
        raise ValueError("pass exactly one of gamma and log_a")
    _buffer(out, "out", B * H * dv, q.dtype, q.device)
    _states(B, H, state_rows(dk, phi), dv, q.device, S=S, z=z)
    _buffer(dev_status, "dev_status", 1, torch.int32, q.device)
    _buffer(log_a, "log_a", B * H, torch.float32, q.device)
    flags = _flags(phi, normalize, True, floor)
    if log_a is not None and (log_a.dtype != torch.float32 or tuple(log_a.shape) != (B, H)):
        raise ValueError(f"log_a must be float32 [B,H] = {(B, H)}")
    with _current(q.device):
        if log_a is None:
            g = _gamma_host(gamma, H)
            st = _load().la_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q),
                                           g.ctypes.data, B, H, dk, dv, flags, float(eps), _ptr(S),
                                           _ptr(z), _ptr(out), _ptr(dev_status), _stream(stream))
            _check(st, "la_recurrent_step")
        else:
            st = _load().la_recurrent_step_gated(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q),
                                                 _ptr(log_a), B, H, dk, dv, flags, float(eps),
                                                 _ptr(S), _ptr(z), _ptr(out), _ptr(dev_status),
                                                 _stream(stream))
            _check(st, "la_recurrent_step_gated")
    return out


def chunk_bwd(q, k, v, dO, gamma=None, *, phi=False, normalize=False, eps=1e-6, S0=None,
              z0=None, dS_T=None, dz_T=None, dq=None, dk=None, dv=None, state_grads=True,
              workspace=None, stream=None, floor=False, log_a=None):
    """Gradients of chunk_fwd for the loss sum(dO * O) + <dS_T, S_T> + <dz_T, z_T>.

    q, k, v, gamma (or log_a), the flags and S0, z0 as in the forward call; dO
    [B,H,T,dv] like v.  Returns (dq, dk, dv, dS0, dz0); dS0 / dz0 are None when
    state_grads is False (dz0 also without the normaliser).  phi="taylor": the
    Taylor feature map (d = 16; the states and their gradients have 273 rows)."""
    normalize = normalize or floor
    B, H, T, dk_ = q.shape
    dv_ = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or dO.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, dO")
    if not (q.dtype == k.dtype == v.dtype == dO.dtype):
        raise TypeError("q, k, v, dO must share one dtype")
    if (gamma is None) == (log_a is None):
        raise ValueError("pass exactly one of gamma and log_a")
    dt = _dtype_code(q)
    dev = q.device
    _inputs(dev, k=k, v=v, dO=dO)
    if log_a is not None and (log_a.dtype != torch.float32 or tuple(log_a.shape) != (B, H, T)):
        raise ValueError(f"log_a must be float32 [B,H,T] = {(B, H, T)}")
    _buffer(log_a, "log_a", B * H * T, torch.float32, dev)
    ds = state_rows(dk_, phi)
    _states(B, H, ds, dv_, dev, S0=S0, z0=z0, dS_T=dS_T, dz_T=dz_T)
    _buffer(dq, "dq", B * H * T * dk_, q.dtype, dev)
    _buffer(dk, "dk", B * H * T * dk_, q.dtype, dev)
    _buffer(dv, "dv", B * H * T * dv_, q.dtype, dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dS0 = torch.empty((B, H, ds, dv_), dtype=torch.float32, device=dev) if state_grads else None
    dz0 = (torch.empty((B, H, ds), dtype=torch.float32, device=dev)
           if state_grads and normalize else None)
    flags = _flags(phi, normalize, True, floor)
    lib = _load()
    with _current(dev):
        need = int(lib.la_bwd_workspace_size(B, H, T, dk_, dv_, dt,
                                             flags | (LA_GATED if log_a is not None else 0)))
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = _workspace(workspace, need, dev)
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(dO), dt)
        rest = (B, H, T, dk_, dv_, flags, float(eps), _ptr(S0), _ptr(z0), _ptr(dS_T), _ptr(dz_T),
                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dS0), _ptr(dz0), _ptr(workspace), ws_bytes,
                None, _stream(stream))
        if log_a is None:
            g = _gamma_host(gamma, H)
            _check(lib.la_chunk_bwd(*args, g.ctypes.data, *rest), "la_chunk_bwd")
        else:
            _check(lib.la_chunk_bwd_gated(*args, _ptr(log_a), *rest), "la_chunk_bwd_gated")
    return dq, dk, dv, dS0, dz0


def host_arena_size(B, H, T, dk, dv, dtype=torch.bfloat16, phi=False, normalize=False,
                    causal=True, chunk=0, pieces=1, floor=False) -> int:
    """Device bytes la_chunk_fwd_host needs for its two slots (la_host_arena_size)."""
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(_load().la_host_arena_size(B, H, T, dk, dv, code, _flags(phi, normalize, causal, floor),
                                          chunk, pieces))


def chunk_fwd_host(q, k, v, gamma, *, phi=False, normalize=False, causal=True, eps=1e-6,
                   S0=None, z0=None, chunk=0, pieces=None, out=None, S_out=None, z_out=None,
                   device="cuda", timing=None, arena=None, floor=False):
    """la_chunk_fwd_host: the chunkwise forward on HOST tensors, copies included.

    q, k, v (and S0, z0) are CPU tensors, pinned for asynchronous copies.  The
    library cuts the batch into `pieces` groups of whole sequences (default: one
    per batch row, at most 8) and pipelines each group's copy in, forward and copy
    out over two streams.  `arena` (a uint8 device tensor of host_arena_size(...)
    bytes) is allocated here when not given.  Returns host (O, S_T, z_T) (z_T when
    normalising or when z_out is given), written into out / S_out / z_out when
    those pinned buffers are passed.  With `timing` (a list), the device
    milliseconds from before the first copy to after the last are appended to it.
    Synchronises before returning.
    """
    normalize = normalize or floor
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for name, t in (("q", q), ("k", k), ("v", v), ("S0", S0), ("z0", z0), ("out", out),
                    ("S_out", S_out), ("z_out", z_out)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host tensor")
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    pin = dict(pin_memory=True)
    ds = state_rows(dk, phi)
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, **pin)
    if S_out is None:
        S_out = torch.empty((B, H, ds, dv), dtype=torch.float32, **pin)
    if z_out is None and normalize:
        z_out = torch.empty((B, H, ds), dtype=torch.float32, **pin)
    host = torch.device("cpu")
    _buffer(out, "out", B * H * T * dv, q.dtype, host)
    _states(B, H, ds, dv, host, S0=S0, z0=z0, S_out=S_out, z_out=z_out)
    n = max(1, min(B, pieces if pieces else min(B, 8)))
    dt = _dtype_code(q)
    flags = _flags(phi, normalize, causal, floor)
    lib = _load()
    g = _gamma_host(gamma, H)
    with torch.cuda.device(dev):
        need = int(lib.la_host_arena_size(B, H, T, dk, dv, dt, flags, int(chunk), n))
        if arena is None:
            arena = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        _buffer(arena, "arena", need, torch.uint8, dev)
        stream = torch.cuda.current_stream(dev)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        st = lib.la_chunk_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), dt, g.ctypes.data, B, H,
                                   T, dk, dv, flags, float(eps),
                                   None if S0 is None else S0.data_ptr(),
                                   None if z0 is None else z0.data_ptr(), out.data_ptr(),
                                   S_out.data_ptr(), None if z_out is None else z_out.data_ptr(),
                                   int(chunk), n, arena.data_ptr(), arena.numel(), None,
                                   stream.cuda_stream or None)
        end.record(stream)
        end.synchronize()
    _check(st, "la_chunk_fwd_host")
    if timing is not None:
        timing.append(start.elapsed_time(end))
    return out, S_out, z_out


__all__ = ["chunk_fwd", "chunk_bwd", "chunk_fwd_noalloc", "recurrent_step", "state_init", "workspace_size", "chunk_fwd_host",
           "host_arena_size",
           "trace_enable", "trace_collect", "debug_set", "debug_options",
           "library", "status_string", "abi_version", "LinAttnError", "LA_PHI_ELU1",
           "LA_NORMALIZE", "LA_NONCAUSAL", "LA_NORM_FLOOR", "LA_GATED", "LA_PHI_TAYLOR", "state_rows"]
