"""The tensor-core kernel's factored per-head decay, checked on the host.

For a chunk of L rows with entry state S (chunkwise form of the "RetNet" page,
"Chunked Recurrent Representation", written out from the recurrence):

  o_i = sum_{j<=i} (q_i . k_j) gamma^(i-j) v_j + gamma^(i+1) q_i S
  S'  = gamma^L S + sum_j gamma^(L-1-j) k_j v_j^T

The kernel computes the same with zeta_j = gamma^(L-1-j) folded into V once:

  V'  = zeta . V,   P_ij = q_i . k_j (j <= i, else 0),
  o_i = gamma^(i+1-L) (P V' + Q (gamma^L S))_i,   S' = gamma^L S + K^T V',

because gamma^(i-j) = gamma^(i+1-L) zeta_j, gamma^(i+1) = gamma^(i+1-L) gamma^L and
sum_j zeta_j k_j v_j^T = K^T (zeta . V).  Here both are checked against the fp64
oracle: the factored form in fp64 (exact up to rounding order), and the factored
form with the kernel's roundings (V', P and the bf16 copy of gamma^L S rounded
to bf16, sums in fp32) within the bf16 tolerance, down to the smallest gamma the
kernel takes it for (gamma^(C-1) = 2^-64) and for the multi-scale retention
heads' gammas.  The per-token decay's factored form (factors about each chunk's
middle exponent, the state carried in tensor memory with a factor the next chunk
takes out) is checked the same way, up to chunks that decay by 2^-160.
"""
import numpy as np
import pytest
import torch

import oracle

C = 128


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def factored(q, k, v, gamma, round_like_kernel=False):
    """One (b, h) sequence chunk by chunk in the factored form; returns O, S_T."""
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv))
    O = np.zeros((T, dv))
    rnd = bf16 if round_like_kernel else (lambda x: x)
    f32 = (lambda x: np.asarray(x, np.float32).astype(np.float64)) if round_like_kernel else (lambda x: x)
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        Q, K, V = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L]
        zeta = gamma ** (L - 1 - np.arange(L, dtype=np.float64))
        Vp = rnd(V * zeta[:, None])
        i = np.arange(L)[:, None]
        j = np.arange(L)[None, :]
        P = rnd(np.where(j <= i, f32(Q @ K.T), 0.0))
        Sg = f32(gamma ** L * S)
        Op = f32(P @ Vp + Q @ rnd(Sg))
        O[c0:c0 + L] = Op * (gamma ** (np.arange(L) + 1.0 - L))[:, None]
        S = f32(Sg + K.T @ Vp)
    return O, S


def case(seed, T, dk, dv, scale):
    rng = np.random.default_rng(seed)
    q = bf16(rng.standard_normal((T, dk)) * scale)
    k = bf16(rng.standard_normal((T, dk)) * scale)
    v = bf16(rng.standard_normal((T, dv)))
    return q, k, v


def rel(a, b):
    return np.abs(a - b).max() / np.abs(b).max()


@pytest.mark.parametrize("gamma", [0.96875, 0.999, 0.8, 2.0 ** (-64 / 127)])
@pytest.mark.parametrize("T", [128, 300, 1])
def test_factored_form_is_the_recurrence(gamma, T):
    q, k, v = case(T, T, 16, 8, 0.25)
    Or, Sr, _ = oracle.recurrent(q[None, None], k[None, None], v[None, None], [gamma])
    O, S = factored(q, k, v, gamma)
    assert rel(O, Or[0, 0]) < 1e-12
    assert rel(S, Sr[0, 0]) < 1e-12


@pytest.mark.parametrize("gamma", [1 - 2.0 ** -5, 1 - 2.0 ** -12, 0.99, 2.0 ** (-64 / 127)])
def test_factored_form_with_kernel_roundings_meets_the_bf16_tolerance(gamma):
    q, k, v = case(7, 700, 64, 32, 64 ** -0.5)
    Or, Sr, _ = oracle.recurrent(q[None, None], k[None, None], v[None, None], [gamma])
    O, S = factored(q, k, v, gamma, round_like_kernel=True)
    assert rel(O, Or[0, 0]) < 2e-2
    assert rel(S, Sr[0, 0]) < 2e-2


def factored_gated(q, k, v, log_a, round_like_kernel=False):
    """The per-token decay in the factored form, about each chunk's middle exponent.

    With b_i = sum_{s<=i} log2 a_s inside the chunk (the "decay, add, read out" loop
    of "Linear Attention, RWKV, and RetNet", 13.3 subsection 4, with a_t per token),
    2^(b_i - b_j) = rho_i zeta_j for rho_i = 2^(b_i - beta), zeta_j = 2^(beta - b_j)
    and beta = (b_0 + b_(L-1)) / 2, and 2^(b_i) q_i S = rho_i q_i (2^beta S).  The
    kernel's tensor memory then holds S' = 2^beta S_in + K^T (zeta . V), which is the
    chunk's exit state times 2^(beta - b_(L-1)): the next chunk's copy of the state
    takes that factor out first (lc below) and multiplies by its own 2^beta after,
    and the exit state takes it out at the end."""
    T, dk = q.shape
    dv = v.shape[1]
    Sp = np.zeros((dk, dv))
    lc = 0.0  # the true state is Sp * 2^lc
    O = np.zeros((T, dv))
    rnd = bf16 if round_like_kernel else (lambda x: x)
    f32 = (lambda x: np.asarray(x, np.float32).astype(np.float64)) if round_like_kernel else (lambda x: x)
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        Q, K, V = q[c0:c0 + L], k[c0:c0 + L], v[c0:c0 + L]
        b = np.cumsum(log_a[c0:c0 + L]) / np.log(2.0)
        beta = 0.5 * (b[0] + b[L - 1])
        Vp = rnd(V * (2.0 ** (beta - b))[:, None])
        i = np.arange(L)[:, None]
        j = np.arange(L)[None, :]
        P = rnd(np.where(j <= i, f32(Q @ K.T), 0.0))
        Sg = f32(f32(Sp * 2.0 ** lc) * 2.0 ** beta)  # two factors, each in range
        Op = f32(P @ Vp + Q @ rnd(Sg))
        O[c0:c0 + L] = Op * (2.0 ** (b - beta))[:, None]
        Sp = f32(Sg + K.T @ Vp)
        lc = b[L - 1] - beta
    return O, Sp * 2.0 ** lc


def gated_case(seed, T, dk, dv, a):
    """Inputs and per-token log decays around log a, a tenth of them halved again."""
    q, k, v = case(seed, T, dk, dv, dk ** -0.5)
    rng = np.random.default_rng(seed + 1)
    log_a = np.log(a) * rng.uniform(0.5, 1.5, T)
    log_a[rng.random(T) < 0.1] += np.log(0.5)
    return q, k, v, np.asarray(log_a, np.float32).astype(np.float64)


def chunk_spread(log_a):
    """Largest decay, in log2 units, from a chunk's first row to its last."""
    b = log_a / np.log(2.0)
    return max(np.sum(b[c0 + 1:c0 + C]) * -1.0 for c0 in range(0, len(b), C))


@pytest.mark.parametrize("a", [0.999, 0.9, 0.6, 0.45])
@pytest.mark.parametrize("T", [128, 300, 1])
def test_centred_factored_form_is_the_gated_recurrence(a, T):
    q, k, v, log_a = gated_case(T, T, 16, 8, a)
    Or, Sr, _ = oracle.recurrent_gated(q[None, None], k[None, None], v[None, None], log_a[None, None])
    O, S = factored_gated(q, k, v, log_a)
    assert rel(O, Or[0, 0]) < 1e-12
    assert rel(S, Sr[0, 0]) < 1e-12


@pytest.mark.parametrize("a", [0.99, 0.8, 0.6, 0.5])
def test_centred_factored_form_with_kernel_roundings_meets_the_bf16_tolerance(a):
    """Up to the bound the kernel takes the factored build for (a chunk's decay from
    its first row to its last at most 2^-160: factors within 2^+-80)."""
    q, k, v, log_a = gated_case(11, 700, 64, 32, a)
    assert chunk_spread(log_a) <= 160
    Or, Sr, _ = oracle.recurrent_gated(q[None, None], k[None, None], v[None, None], log_a[None, None])
    O, S = factored_gated(q, k, v, log_a, round_like_kernel=True)
    assert rel(O, Or[0, 0]) < 2e-2
    assert rel(S, Sr[0, 0]) < 2e-2
