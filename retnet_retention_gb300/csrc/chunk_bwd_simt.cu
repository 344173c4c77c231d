// Backward pass (gradients) of the causal chunkwise forward, on the CUDA cores
// in fp32.
//
// "Linear attention" (zerotofrontier 21.2), "Decoding, training, and what each
// costs": the gradients are cumulative sums too, running forward in time for
// the queries and backward in time for the keys and values, so no state is
// stored.  Chunked like the forward ("Chunked Recurrent Representation",
// "RetNet" page): inside a chunk the parallel form, across chunks a carried
// state.  For the loss L = sum_t do_t . o_t + <dS_T, S_T> + <dz_T, z_T>, a
// chunk of L rows with local indices i, j, D_ij = gamma^(i-j) (j <= i),
// xi_i = gamma^(i+1), zeta_j = gamma^(L-1-j) (or the per-token decay's
// cumulative-log forms, as in the forward kernels):
//
//   forward sweep (role 0), entry state S, z:
//     A_ij = D_ij q~_i . k~_j,   n_i = sum_j A_ij v_j + xi_i q~_i S
//     u_i  = sum_j A_ij + xi_i q~_i . z,   den_i = u_i + eps or max(|u_i|, 1)
//     dn_i = do_i / den_i,   du_i = -(do_i . n_i) / den_i^2 * dden/du
//     P_ij = D_ij (dn_i . v_j + du_i)
//     dq~_i = sum_j P_ij k~_j + xi_i (S dn_i + du_i z)
//   backward sweep (role 1), G = dL/dS and Gz = dL/dz at the chunk's end:
//     dv_j  = sum_{i>=j} A_ij dn_i + zeta_j k~_j G
//     dk~_j = sum_{i>=j} P_ij q~_i + zeta_j (G v_j + Gz)
//     G <- gamma^L G + sum_i xi_i q~_i^T dn_i,  Gz <- gamma^L Gz + sum_i xi_i du_i q~_i
//   and dS_0 = G, dz_0 = Gz at the start.  phi: dq = dq~ * phi'(q) with
//   phi'(x) = min(1, phi(x)) for phi = elu + 1.
//
// Without the normaliser (den = 1, du = 0) the two sweeps are independent and
// run as one launch, one CTA per (b, h) and sweep; with it the backward sweep
// reads the forward sweep's den_i and du_i (per token, in the workspace), so
// the forward sweep runs first.  One CTA holds the whole d_k x d_v state of its
// (b, h) in shared memory (d_k, d_v <= 128).
#include "launch.h"
#include "trace.h"

namespace la {

namespace {

constexpr int kThreads = 256;

struct BwdSmem {  // offsets in floats
    int q, k, v, g, n, a, p, s, z, den, du, pw, cum, xw, total;
};

__host__ __device__ inline BwdSmem bwd_layout(int C, int dk, int dv) {
    BwdSmem L;
    const int ldk = dk + 1, ldv = dv + 1, lda = C + 1;
    L.q = 0;
    L.k = L.q + C * ldk;
    L.v = L.k + C * ldk;
    L.g = L.v + C * ldv;   // dO, then dn = dO / den
    L.n = L.g + C * ldv;   // n_i (forward sweep)
    L.a = L.n + C * ldv;
    L.p = L.a + C * lda;
    L.s = L.p + C * lda;   // S (forward sweep) or G (backward sweep), rows dv + 1 apart
    L.z = L.s + dk * ldv;  // z or Gz
    L.den = L.z + dk;
    L.du = L.den + C;
    L.pw = L.du + C;
    L.cum = L.pw + C + 2;
    L.xw = L.cum + C;
    L.total = L.xw + C;
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_bwd_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ S0, const float* __restrict__ z0,
    const float* __restrict__ dST, const float* __restrict__ dzT, T* __restrict__ dQ,
    T* __restrict__ dK, T* __restrict__ dV, float* __restrict__ dS0, float* __restrict__ dz0,
    float* __restrict__ stats, int H, int T_len, int dk, int dv, int C, int phi, int normalize,
    float eps, int role0, const float* __restrict__ log_a, const __grid_constant__ KernelGammas g) {
    extern __shared__ float smem[];
    const BwdSmem lay = bwd_layout(C, dk, dv);
    float* Qs = smem + lay.q;
    float* Ks = smem + lay.k;
    float* Vs = smem + lay.v;
    float* Gs = smem + lay.g;
    float* Ns = smem + lay.n;
    float* As = smem + lay.a;
    float* Ps = smem + lay.p;
    float* Ss = smem + lay.s;
    float* zs = smem + lay.z;
    float* den = smem + lay.den;
    float* du = smem + lay.du;
    float* pw = smem + lay.pw;
    float* cum = smem + lay.cum;
    float* xw = smem + lay.xw;
    const int ldk = dk + 1, ldv = dv + 1, lda = C + 1, lds = dv + 1;

    const int bh = blockIdx.x;
    const int role = role0 + (int)blockIdx.y;  // 0: forward sweep (dq), 1: backward sweep (dk, dv)
    const int h = bh % H;
    const int tid = threadIdx.x;
    const float l2g = g.log2g[h];
    const size_t qk_base = (size_t)bh * T_len * dk;
    const size_t v_base = (size_t)bh * T_len * dv;
    const int n_chunks = (T_len + C - 1) / C;

    for (int n = tid; n <= C; n += kThreads) pw[n] = gamma_pow(l2g, (float)n);
    // entry state: S0, z0 (forward sweep) or dS_T, dz_T (backward sweep)
    const float* s_in = role == 0 ? S0 : dST;
    const float* z_in = role == 0 ? z0 : dzT;
    for (int idx = tid; idx < dk * dv; idx += kThreads)
        Ss[(idx / dv) * lds + idx % dv] = s_in ? s_in[(size_t)bh * dk * dv + idx] : 0.f;
    for (int d = tid; d < dk; d += kThreads) zs[d] = z_in ? z_in[(size_t)bh * dk + d] : 0.f;
    __syncthreads();

    for (int cc = 0; cc < n_chunks; ++cc) {
        const int c = role == 0 ? cc : n_chunks - 1 - cc;
        const int t0 = c * C;
        const int L = min(C, T_len - t0);
        // tiles: phi(Q), phi(K), V, dO (rows >= L zero)
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            const int i = idx / dk, d = idx % dk;
            float x = 0.f, y = 0.f;
            if (i < L) {
                const size_t gi = qk_base + (size_t)(t0 + i) * dk + d;
                x = load_elem(Q, gi);
                y = load_elem(K, gi);
                if (phi) {
                    x = phi_elu1(x);
                    y = phi_elu1(y);
                }
            }
            Qs[i * ldk + d] = x;
            Ks[i * ldk + d] = y;
        }
        for (int idx = tid; idx < C * dv; idx += kThreads) {
            const int i = idx / dv, cc2 = idx % dv;
            float x = 0.f, y = 0.f;
            if (i < L) {
                const size_t gi = v_base + (size_t)(t0 + i) * dv + cc2;
                x = load_elem(V, gi);
                y = load_elem(dO, gi);
            }
            Vs[i * ldv + cc2] = x;
            Gs[i * ldv + cc2] = y;
        }
        if (log_a && tid == 0) {  // b_i = sum_{s<=i} log a_s, in log2 units
            float acc = 0.f;
            for (int i = 0; i < L; ++i) {
                acc += log_a[(size_t)bh * T_len + t0 + i] * 1.44269504088896341f;
                cum[i] = acc;
            }
        }
        if (role == 1 && normalize)
            for (int i = tid; i < L; i += kThreads) {
                den[i] = stats[((size_t)bh * T_len + t0 + i) * 2];
                du[i] = stats[((size_t)bh * T_len + t0 + i) * 2 + 1];
            }
        __syncthreads();
        float* zeta = pw;  // per-token decay: zeta_j in pw, xi_i in xw
        if (log_a) {
            for (int i = tid; i < L; i += kThreads) {
                xw[i] = exp2f(cum[i]);
                pw[i] = exp2f(cum[L - 1] - cum[i]);
            }
            __syncthreads();
        }
        auto dmask = [&](int i, int j) { return log_a ? exp2f(cum[i] - cum[j]) : pw[i - j]; };
        auto xi = [&](int i) { return log_a ? xw[i] : pw[i + 1]; };
        auto zt = [&](int j) { return log_a ? zeta[j] : pw[L - 1 - j]; };
        const float gL = log_a ? exp2f(cum[L - 1]) : pw[L];
        // Register tiles: a thread computes 4 output rows x 2 columns (c = 64 g + slot
        // and c + 32), so each shared-memory operand it loads feeds 2 or 4 FMAs; the
        // 32 items of a warp share their rows (broadcast loads) and take consecutive
        // columns.  Every output keeps its summation order.
        auto tiles = [&](int R, int D, auto&& body) {
            const int ng = (D + 63) >> 6;
            const int items = ((R + 3) >> 2) * ng * 32;
            for (int item = tid; item < items; item += kThreads) {
                const int slot = item & 31, rest = item >> 5;
                const int c0 = 64 * (rest % ng) + slot;
                body((rest / ng) * 4, c0, c0 + 32);
            }
        };

        // A_ij = D_ij q~_i . k~_j (j <= i): tiles of 4 rows i and one column j
        for (int item = tid; item < ((L + 3) >> 2) * 32; item += kThreads) {
            const int j = item & 31, i0 = (item >> 5) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (j < L && j <= i0 + 3) {
                const float* kj = Ks + j * ldk;
                for (int d = 0; d < dk; ++d) {
                    const float kv = kj[d];
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[r] = fmaf(Qs[(i0 + r) * ldk + d], kv, acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                if (i < L && j < L) As[i * lda + j] = j <= i ? acc[r] * dmask(i, j) : 0.f;
            }
        }
        __syncthreads();
        if (role == 0) {
            if (normalize) {
                // n_i = sum_j A_ij v_j + xi_i q~_i S  (A_ij = 0 above the diagonal)
                tiles(L, dv, [&](int i0, int c0, int c1) {
                    const int a0 = c0 < dv ? c0 : 0, a1 = c1 < dv ? c1 : 0;
                    float in[4][2] = {}, it[4][2] = {};
                    const int jmax = min(i0 + 3, L - 1);
                    for (int j = 0; j <= jmax; ++j) {
                        const float x0 = Vs[j * ldv + a0], x1 = Vs[j * ldv + a1];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float a = As[(i0 + r) * lda + j];
                            in[r][0] = fmaf(a, x0, in[r][0]);
                            in[r][1] = fmaf(a, x1, in[r][1]);
                        }
                    }
                    for (int d = 0; d < dk; ++d) {
                        const float s0 = Ss[d * lds + a0], s1 = Ss[d * lds + a1];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float q = Qs[(i0 + r) * ldk + d];
                            it[r][0] = fmaf(q, s0, it[r][0]);
                            it[r][1] = fmaf(q, s1, it[r][1]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int i = i0 + r;
                        if (i >= L) continue;
                        if (c0 < dv) Ns[i * ldv + c0] = in[r][0] + xi(i) * it[r][0];
                        if (c1 < dv) Ns[i * ldv + c1] = in[r][1] + xi(i) * it[r][1];
                    }
                });
                __syncthreads();
                // den_i, du_i (one warp per row: the sums over d_k and d_v)
                const int warp = tid >> 5, lane = tid & 31;
                for (int i = warp; i < L; i += kThreads / 32) {
                    float r = 0.f, qz = 0.f, don = 0.f;
                    for (int j = lane; j <= i; j += 32) r += As[i * lda + j];
                    for (int d = lane; d < dk; d += 32) qz = fmaf(Qs[i * ldk + d], zs[d], qz);
                    for (int cc2 = lane; cc2 < dv; cc2 += 32)
                        don = fmaf(Gs[i * ldv + cc2], Ns[i * ldv + cc2], don);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        r += __shfl_xor_sync(0xffffffffu, r, off);
                        qz += __shfl_xor_sync(0xffffffffu, qz, off);
                        don += __shfl_xor_sync(0xffffffffu, don, off);
                    }
                    if (lane == 0) {
                        const float u = r + xi(i) * qz;
                        const float dd = norm_den(u, normalize, eps);
                        const float dd_du = normalize == 2 ? (fabsf(u) > 1.f ? (u > 0.f ? 1.f : -1.f) : 0.f)
                                                           : 1.f;
                        den[i] = dd;
                        du[i] = -don / (dd * dd) * dd_du;
                        stats[((size_t)bh * T_len + t0 + i) * 2] = dd;
                        stats[((size_t)bh * T_len + t0 + i) * 2 + 1] = du[i];
                    }
                }
                __syncthreads();
            }
        }
        // dn_i = dO_i / den_i (in place)
        if (normalize) {
            for (int idx = tid; idx < L * dv; idx += kThreads) {
                const int i = idx / dv, cc2 = idx % dv;
                Gs[i * ldv + cc2] /= den[i];
            }
            __syncthreads();
        }
        // P_ij = D_ij (dn_i . v_j + du_i)  (j <= i): tiles of 4 rows i and one column j
        for (int item = tid; item < ((L + 3) >> 2) * 32; item += kThreads) {
            const int j = item & 31, i0 = (item >> 5) * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (j < L && j <= i0 + 3) {
                const float* vj = Vs + j * ldv;
                for (int cc2 = 0; cc2 < dv; ++cc2) {
                    const float vv = vj[cc2];
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[r] = fmaf(Gs[(i0 + r) * ldv + cc2], vv, acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                if (i < L && j < L)
                    Ps[i * lda + j] = j <= i ? (acc[r] + (normalize ? du[i] : 0.f)) * dmask(i, j) : 0.f;
            }
        }
        __syncthreads();
        if (role == 0) {
            // dq~_i = sum_j P_ij k~_j + xi_i (S dn_i + du_i z);  dq = dq~ * phi'(q)
            tiles(L, dk, [&](int i0, int c0, int c1) {
                const int a0 = c0 < dk ? c0 : 0, a1 = c1 < dk ? c1 : 0;
                float in[4][2] = {}, it[4][2] = {};
                const int jmax = min(i0 + 3, L - 1);
                for (int j = 0; j <= jmax; ++j) {
                    const float k0 = Ks[j * ldk + a0], k1 = Ks[j * ldk + a1];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float pp = Ps[(i0 + r) * lda + j];
                        in[r][0] = fmaf(pp, k0, in[r][0]);
                        in[r][1] = fmaf(pp, k1, in[r][1]);
                    }
                }
                for (int cc2 = 0; cc2 < dv; ++cc2) {
                    const float s0 = Ss[a0 * lds + cc2], s1 = Ss[a1 * lds + cc2];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float gg = Gs[(i0 + r) * ldv + cc2];
                        it[r][0] = fmaf(s0, gg, it[r][0]);
                        it[r][1] = fmaf(s1, gg, it[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = i0 + r;
                    if (i >= L) continue;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int d = e ? c1 : c0;
                        if (d >= dk) continue;
                        float inter = it[r][e];
                        if (normalize) inter = fmaf(du[i], zs[d], inter);
                        float v = in[r][e] + xi(i) * inter;
                        if (phi) v *= fminf(1.f, Qs[i * ldk + d]);
                        store_elem(dQ, qk_base + (size_t)(t0 + i) * dk + d, v);
                    }
                }
            });
            __syncthreads();
            // S = gamma^L S + sum_j zeta_j k~_j^T v_j ; z likewise
            tiles(dk, dv, [&](int d0, int c0, int c1) {
                const int a0 = c0 < dv ? c0 : 0, a1 = c1 < dv ? c1 : 0;
                float u[4][2] = {};
                for (int j = 0; j < L; ++j) {
                    const float x0 = Vs[j * ldv + a0], x1 = Vs[j * ldv + a1], zj = zt(j);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float kk = zj * Ks[j * ldk + d0 + r];
                        u[r][0] = fmaf(kk, x0, u[r][0]);
                        u[r][1] = fmaf(kk, x1, u[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int d = d0 + r;
                    if (c0 < dv) Ss[d * lds + c0] = fmaf(gL, Ss[d * lds + c0], u[r][0]);
                    if (c1 < dv) Ss[d * lds + c1] = fmaf(gL, Ss[d * lds + c1], u[r][1]);
                }
            });
            for (int d = tid; d < dk; d += kThreads) {
                float u = 0.f;
                for (int j = 0; j < L; ++j) u = fmaf(zt(j), Ks[j * ldk + d], u);
                zs[d] = fmaf(gL, zs[d], u);
            }
            __syncthreads();
        } else {
            // dv_j = sum_{i>=j} A_ij dn_i + zeta_j k~_j G
            tiles(L, dv, [&](int j0, int c0, int c1) {
                const int a0 = c0 < dv ? c0 : 0, a1 = c1 < dv ? c1 : 0;
                float in[4][2] = {}, it[4][2] = {};
                for (int i = j0; i < L; ++i) {  // A_ij = 0 for i < j
                    const float g0 = Gs[i * ldv + a0], g1 = Gs[i * ldv + a1];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float a = As[i * lda + j0 + r];
                        in[r][0] = fmaf(a, g0, in[r][0]);
                        in[r][1] = fmaf(a, g1, in[r][1]);
                    }
                }
                for (int d = 0; d < dk; ++d) {
                    const float s0 = Ss[d * lds + a0], s1 = Ss[d * lds + a1];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float kk = Ks[(j0 + r) * ldk + d];
                        it[r][0] = fmaf(kk, s0, it[r][0]);
                        it[r][1] = fmaf(kk, s1, it[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int j = j0 + r;
                    if (j >= L) continue;
                    if (c0 < dv) store_elem(dV, v_base + (size_t)(t0 + j) * dv + c0, in[r][0] + zt(j) * it[r][0]);
                    if (c1 < dv) store_elem(dV, v_base + (size_t)(t0 + j) * dv + c1, in[r][1] + zt(j) * it[r][1]);
                }
            });
            // dk~_j = sum_{i>=j} P_ij q~_i + zeta_j (G v_j + Gz);  dk = dk~ * phi'(k)
            tiles(L, dk, [&](int j0, int c0, int c1) {
                const int a0 = c0 < dk ? c0 : 0, a1 = c1 < dk ? c1 : 0;
                float in[4][2] = {}, it[4][2] = {};
                for (int i = j0; i < L; ++i) {  // P_ij = 0 for i < j
                    const float q0 = Qs[i * ldk + a0], q1 = Qs[i * ldk + a1];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float pp = Ps[i * lda + j0 + r];
                        in[r][0] = fmaf(pp, q0, in[r][0]);
                        in[r][1] = fmaf(pp, q1, in[r][1]);
                    }
                }
                for (int cc2 = 0; cc2 < dv; ++cc2) {
                    const float s0 = Ss[a0 * lds + cc2], s1 = Ss[a1 * lds + cc2];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float vv = Vs[(j0 + r) * ldv + cc2];
                        it[r][0] = fmaf(s0, vv, it[r][0]);
                        it[r][1] = fmaf(s1, vv, it[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int j = j0 + r;
                    if (j >= L) continue;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int d = e ? c1 : c0;
                        if (d >= dk) continue;
                        float inter = it[r][e];
                        if (normalize) inter += zs[d];
                        float v = in[r][e] + zt(j) * inter;
                        if (phi) v *= fminf(1.f, Ks[j * ldk + d]);
                        store_elem(dK, qk_base + (size_t)(t0 + j) * dk + d, v);
                    }
                }
            });
            __syncthreads();
            // G = gamma^L G + sum_i xi_i q~_i^T dn_i ;  Gz = gamma^L Gz + sum_i xi_i du_i q~_i
            tiles(dk, dv, [&](int d0, int c0, int c1) {
                const int a0 = c0 < dv ? c0 : 0, a1 = c1 < dv ? c1 : 0;
                float u[4][2] = {};
                for (int i = 0; i < L; ++i) {
                    const float g0 = Gs[i * ldv + a0], g1 = Gs[i * ldv + a1], x = xi(i);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float qq = x * Qs[i * ldk + d0 + r];
                        u[r][0] = fmaf(qq, g0, u[r][0]);
                        u[r][1] = fmaf(qq, g1, u[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int d = d0 + r;
                    if (c0 < dv) Ss[d * lds + c0] = fmaf(gL, Ss[d * lds + c0], u[r][0]);
                    if (c1 < dv) Ss[d * lds + c1] = fmaf(gL, Ss[d * lds + c1], u[r][1]);
                }
            });
            if (normalize)
                for (int d = tid; d < dk; d += kThreads) {
                    float u = 0.f;
                    for (int i = 0; i < L; ++i) u = fmaf(xi(i) * du[i], Qs[i * ldk + d], u);
                    zs[d] = fmaf(gL, zs[d], u);
                }
            __syncthreads();
        }
    }
    if (role == 1) {  // gradients of the initial state
        if (dS0)
            for (int idx = tid; idx < dk * dv; idx += kThreads)
                dS0[(size_t)bh * dk * dv + idx] = Ss[(idx / dv) * lds + idx % dv];
        if (dz0)
            for (int d = tid; d < dk; d += kThreads) dz0[(size_t)bh * dk + d] = zs[d];
    }
}

}  // namespace

int bwd_chunk_len(int dk, int dv) {
    int C = 32;
    while (C > 8 && (size_t)bwd_layout(C, dk, dv).total * 4 > 227 * 1024) C >>= 1;
    return C;
}

size_t bwd_workspace_bytes(int B, int H, int T, bool normalize) {
    return normalize ? (size_t)B * H * T * 2 * sizeof(float) : 0;
}

cudaError_t launch_chunk_bwd_simt(const BwdArgs& a, const KernelGammas& g, cudaStream_t s) {
    const int C = bwd_chunk_len(a.dk, a.dv);
    const size_t smem = (size_t)bwd_layout(C, a.dk, a.dv).total * sizeof(float);
    const unsigned nbh = (unsigned)((size_t)a.B * a.H);
    const int nm = norm_mode(a.normalize, a.floor_norm);
    float* stats = static_cast<float*>(a.workspace);
    cudaError_t e = cudaSuccess;
    auto launch = [&](auto kern, auto cast, int role0, unsigned roles) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return;
        TraceScope trace(roles == 2 ? "chunk_bwd_simt_kernel"
                         : role0 == 0 ? "chunk_bwd_simt_kernel/dq" : "chunk_bwd_simt_kernel/dkdv",
                         s);
        kern<<<dim3(nbh, roles), kThreads, smem, s>>>(
            cast(a.Q), cast(a.K), cast(a.V), cast(a.dO), a.S0, a.z0, a.dS_T, a.dz_T, cast(a.dQ),
            cast(a.dK), cast(a.dV), a.dS0, a.dz0, stats, a.H, a.T, a.dk, a.dv, C, a.phi, nm,
            a.eps, role0, a.log_a, g);
        e = cudaGetLastError();
    };
    auto run = [&](auto kern, auto cast) {
        if (nm == 0) {
            launch(kern, cast, 0, 2);  // the two sweeps are independent
        } else {
            launch(kern, cast, 0, 1);  // the backward sweep reads the forward sweep's den, du
            if (e == cudaSuccess) launch(kern, cast, 1, 1);
        }
    };
    if (a.bf16)
        run(chunk_bwd_simt_kernel<__nv_bfloat16>,
            [](const void* p) { return (__nv_bfloat16*)const_cast<void*>(p); });
    else
        run(chunk_bwd_simt_kernel<float>, [](const void* p) { return (float*)const_cast<void*>(p); });
    return e;
}

}  // namespace la
