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
// run side by side; with it the backward sweep reads the forward sweep's den_i
// and du_i (per token, in the workspace), so the forward sweep runs first.  One
// CTA holds the whole d_k x d_v state of its (b, h) in shared memory (d_k, d_v
// <= 128).
//
// Segments: so that every SM holds several CTAs, each sequence is cut into P
// segments of whole chunks.  Each segment's own contribution (forward: S and z
// from zero over the segment; backward: G and Gz from zero, i.e. the gradient of
// the segment's own outputs with respect to the state entering it) comes from a
// weighted product over its tokens (bwd_state_gemm_kernel, d_k and d_v in
// {64, 128}) or a state-only pass of the chunked kernel, a scan folds them into
// entry states (forward:
// S_entry(q+1) = d(q) S_entry(q) + agg(q) from S_0; backward: G_end(q) =
// d(q+1) G_end(q+1) + gagg(q+1) from dS_T; d(q) the state's decay over segment
// q), and the full sweeps run every segment from its entry state.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "launch.h"
#include "trace.h"

namespace la {

namespace {

constexpr int kThreads = 256;

// The segment plan of one launch (see the header).
struct BwdSeg {
    int n_seg;          // segments per sequence
    int seg_chunks;     // chunks (of C tokens) per segment
    int state_only;     // 1: only the segment's own state contribution
    const float* S_ent; // full forward sweep: entry states [BH][n_seg][dk][dv] (null: S0)
    const float* z_ent; // [BH][n_seg][dk] (null: z0)
    const float* G_ent; // full backward sweep: G at each segment's end (null: dS_T)
    const float* Gz_ent;
    float* agg;         // state-only forward sweep: [BH][n_seg][dk][dv]
    float* zagg;        // state-only forward sweep: [BH][n_seg][dk]
    float* agg1;        // state-only backward sweep: the same for G and Gz
    float* zagg1;
    float* seg_l2;      // state-only forward sweep, per-token decay: the segment's
                        // total log2 decay [BH][n_seg]
};

template <typename T>
struct Raw8;  // 8 consecutive input elements in registers
template <>
struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ void load(const __nv_bfloat16* p) { u = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ void to_f32(float (&x)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w[e] << 16);
            x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ void load(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ void to_f32(float (&x)[8]) const {
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w;
        x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
    }
};

struct BwdSmem {  // offsets in floats
    int q, k, v, g, n, a, p, s, z, den, du, pw, cum, xw, tq, total;
};

// dk: the state's rows (the feature dimension: 1 + d + d^2 with the Taylor map);
// with the Taylor map a [C][dk + 1] buffer holds the gradient of a chunk's features
// before the chain rule takes it back to the raw d columns.
__host__ __device__ inline BwdSmem bwd_layout(int C, int dk, int dv, bool taylor = false) {
    BwdSmem L;
    const int ldk = dk + 1, ldv = dv + 1, lda = C + 1;
    L.q = 0;
    L.k = L.q + C * ldk;
    L.v = L.k + C * ldk;
    L.g = L.v + C * ldv;   // dO, then dn = dO / den
    // S dO_i (forward sweep with the normaliser; in the tq buffer with the Taylor
    // map); the decayed copy for the state update
    L.n = L.g + C * ldv;
    L.a = L.n + C * (taylor ? dv + 4 : std::max(dv + 4, ldk));
    L.p = L.a + C * lda;
    L.s = L.p + C * lda;   // S (forward sweep) or G (backward sweep), rows dv + 1 apart
    L.z = L.s + dk * ldv;  // z or Gz
    L.den = L.z + dk;
    L.du = L.den + C;
    L.pw = L.du + C;
    L.cum = L.pw + C + 2;
    L.xw = L.cum + C;
    L.tq = L.xw + C;
    L.total = L.tq + (taylor ? C * ldk : 0);
    return L;
}

// DKc, DVc, CC: d_k, d_v and the chunk length fixed at compile time (0: the
// arguments), so that the loops over them unroll and their index arithmetic folds.
// Registers: 64 a thread for the run-time shapes (four CTAs an SM), 80 for
// d_k = d_v = 64 (three CTAs, as many as its shared memory allows), no limit for
// 128 (one CTA).
template <typename T, int DKc = 0, int DVc = 0, int CC = 0>
__global__ void __launch_bounds__(kThreads, DKc == 0 ? 4 : DKc == 64 && DVc == 64 ? 3 : 1) chunk_bwd_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ S0, const float* __restrict__ z0,
    const float* __restrict__ dST, const float* __restrict__ dzT, T* __restrict__ dQ,
    T* __restrict__ dK, T* __restrict__ dV, float* __restrict__ dS0, float* __restrict__ dz0,
    float* __restrict__ stats, int H, int T_len, int dk_arg, int dv_arg, int C_arg, int phi,
    int normalize, float eps, int role0, const float* __restrict__ log_a,
    const __grid_constant__ KernelGammas g, const __grid_constant__ BwdSeg sg, int d_in, int taylor) {
    const int dk = DKc ? DKc : dk_arg;
    const int dv = DVc ? DVc : dv_arg;
    const int C = CC ? CC : C_arg;
    // fixed shapes: rows of Q, K, V and dO loaded 8 elements at a time (16 bytes
    // of bf16; the host checks the alignment)
    constexpr bool kVec = DKc > 0 && DVc > 0 && DKc % 8 == 0 && DVc % 8 == 0;
    extern __shared__ float smem[];
    const BwdSmem lay = bwd_layout(C, dk, dv, taylor != 0);
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
    float* TQ = smem + lay.tq;  // Taylor map: a chunk's feature gradients, rows ldk apart
    const int ldk = dk + 1, ldv = dv + 1, lda = C + 1, lds = dv + 1;
    const float kR2 = 0.70710678118654752f;  // 1 / sqrt 2

    const int bh = blockIdx.x / sg.n_seg;
    const int seg = blockIdx.x % sg.n_seg;
    const size_t sidx = (size_t)bh * sg.n_seg + seg;  // this unit's entry / contribution slot
    const int role = role0 + (int)blockIdx.y;  // 0: forward sweep (dq), 1: backward sweep (dk, dv)
    const bool st_only = sg.state_only != 0;
    const int h = bh % H;
    const int tid = threadIdx.x;
    const float l2g = g.log2g[h];
    const size_t qk_base = (size_t)bh * T_len * d_in;  // rows of Q, K (and dQ, dK): d_in wide
    const size_t v_base = (size_t)bh * T_len * dv;
    const int n_chunks = (T_len + C - 1) / C;
    const int cb = seg * sg.seg_chunks;
    const int ce = min(n_chunks, cb + sg.seg_chunks);

    for (int n = tid; n <= C; n += kThreads) pw[n] = gamma_pow(l2g, (float)n);
    // entry state: S0, z0 or the segment's entry (forward sweep); dS_T, dz_T or the
    // state's gradient at the segment's end (backward sweep); zero for a state-only pass
    const float* s_in = nullptr;
    const float* z_in = nullptr;
    if (!st_only) {
        if (role == 0) {
            s_in = sg.S_ent ? sg.S_ent + sidx * dk * dv : (S0 ? S0 + (size_t)bh * dk * dv : nullptr);
            z_in = sg.z_ent ? sg.z_ent + sidx * dk : (z0 ? z0 + (size_t)bh * dk : nullptr);
        } else {
            s_in = sg.G_ent ? sg.G_ent + sidx * dk * dv : (dST ? dST + (size_t)bh * dk * dv : nullptr);
            z_in = sg.Gz_ent ? sg.Gz_ent + sidx * dk : (dzT ? dzT + (size_t)bh * dk : nullptr);
        }
    }
    for (int idx = tid; idx < dk * dv; idx += kThreads)
        Ss[(idx / dv) * lds + idx % dv] = s_in ? s_in[idx] : 0.f;
    for (int d = tid; d < dk; d += kThreads) zs[d] = z_in ? z_in[d] : 0.f;
    float seg_lam = 0.f;  // per-token decay: the segment's total log2 decay (thread 0)
    // The Taylor map's transpose Jacobian for rows 0 .. L-1 of a chunk: x_c sits in
    // feature 1 + c and in the outer product's row c and column c (each over
    // sqrt 2), so dx_c = dF_(1+c) + (sum_b (dF_(1+d_in+c*d_in+b) + dF_(1+d_in+b*d_in+c))
    // x_b) / sqrt 2, with x the raw row (features 1 .. d_in of F).
    auto taylor_back = [&](const float* dF, const float* F, T* out, int L, int t0) {
        for (int idx = tid; idx < L * d_in; idx += kThreads) {
            const int i = idx / d_in, c = idx % d_in;
            const float* gr = dF + i * ldk;
            const float* xr = F + i * ldk + 1;
            float acc = 0.f;
            for (int b = 0; b < d_in; ++b)
                acc = fmaf(gr[1 + d_in + c * d_in + b] + gr[1 + d_in + b * d_in + c], xr[b], acc);
            store_elem(out, qk_base + (size_t)(t0 + i) * d_in + c, fmaf(kR2, acc, gr[1 + c]));
        }
    };
    __syncthreads();

    for (int cc = cb; cc < ce; ++cc) {
        const int c = role == 0 ? cc : ce - 1 - (cc - cb);
        const int t0 = c * C;
        const int L = min(C, T_len - t0);
        // tiles: phi(Q), phi(K), V, dO (rows >= L zero); a state-only pass reads
        // K and V (forward sweep) or Q and dO (backward sweep) only
        const bool need_qg = !st_only || role == 1, need_kv = !st_only || role == 0;
        if constexpr (kVec) {  // Q and K 8 elements a load
            for (int idx = tid; idx < C * dk / 8; idx += kThreads) {
                const int i = idx / (dk / 8), d0 = (idx % (dk / 8)) * 8;
                float x[8], y[8];
                const size_t gi = qk_base + (size_t)(t0 + i) * dk + d0;
                Raw8<T> rx, ry;
                if (i < L && need_qg) rx.load(Q + gi);
                if (i < L && need_kv) ry.load(K + gi);
                rx.to_f32(x);
                ry.to_f32(y);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float xv = x[e], yv = y[e];
                    if (phi) {
                        xv = phi_elu1(xv);
                        yv = phi_elu1(yv);
                    }
                    Qs[i * ldk + d0 + e] = i < L && need_qg ? xv : 0.f;
                    Ks[i * ldk + d0 + e] = i < L && need_kv ? yv : 0.f;
                }
            }
        }
        for (int idx = tid; idx < (kVec ? 0 : C * dk); idx += kThreads) {
            const int i = idx / dk, d = idx % dk;
            float x = 0.f, y = 0.f;
            if (i < L && taylor) {
                // feature d of the row: 1, then x_c, then x_a x_b / sqrt 2 (a-major)
                const size_t r0 = qk_base + (size_t)(t0 + i) * d_in;
                if (d == 0) {
                    x = need_qg ? 1.f : 0.f;
                    y = need_kv ? 1.f : 0.f;
                } else if (d <= d_in) {
                    if (need_qg) x = load_elem(Q, r0 + d - 1);
                    if (need_kv) y = load_elem(K, r0 + d - 1);
                } else {
                    const int a = (d - 1 - d_in) / d_in, b = (d - 1 - d_in) % d_in;
                    if (need_qg) x = load_elem(Q, r0 + a) * load_elem(Q, r0 + b) * kR2;
                    if (need_kv) y = load_elem(K, r0 + a) * load_elem(K, r0 + b) * kR2;
                }
            } else if (i < L) {
                const size_t gi = qk_base + (size_t)(t0 + i) * dk + d;
                if (need_qg) x = load_elem(Q, gi);
                if (need_kv) y = load_elem(K, gi);
                if (phi) {
                    x = phi_elu1(x);
                    y = phi_elu1(y);
                }
            }
            Qs[i * ldk + d] = x;
            Ks[i * ldk + d] = y;
        }
        if constexpr (kVec) {  // V and dO 8 elements a load
            for (int idx = tid; idx < C * dv / 8; idx += kThreads) {
                const int i = idx / (dv / 8), c0 = (idx % (dv / 8)) * 8;
                float x[8], y[8];
                const size_t gi = v_base + (size_t)(t0 + i) * dv + c0;
                Raw8<T> rx, ry;
                if (i < L && need_kv) rx.load(V + gi);
                if (i < L && need_qg) ry.load(dO + gi);
                rx.to_f32(x);
                ry.to_f32(y);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    Vs[i * ldv + c0 + e] = i < L && need_kv ? x[e] : 0.f;
                    Gs[i * ldv + c0 + e] = i < L && need_qg ? y[e] : 0.f;
                }
            }
        }
        for (int idx = tid; idx < (kVec ? 0 : C * dv); idx += kThreads) {
            const int i = idx / dv, cc2 = idx % dv;
            float x = 0.f, y = 0.f;
            if (i < L) {
                const size_t gi = v_base + (size_t)(t0 + i) * dv + cc2;
                if (need_kv) x = load_elem(V, gi);
                if (need_qg) y = load_elem(dO, gi);
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
        if (log_a && tid == 0) seg_lam += cum[L - 1];
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
        // Fixed shapes: the state's update Ss = gL Ss + X^T (w . Y) over the chunk's
        // rows (X = K~, Y = V, w = zeta forward; X = Q~, Y = dn, w = xi backward).
        // w . Y goes to the n buffer with rows d_v + 4 apart (16-byte aligned), then
        // thread t takes the 4 x 4 block at rows 4 (t / (d_v / 4)) and columns
        // 4 (t % (d_v / 4)): per row of the chunk one 16-byte load of w . Y and four
        // loads of X that the warp's lanes share, for 16 FMAs.
        auto state_update = [&](const float* X, const float* Y, auto&& w, float gL) {
            if constexpr (kVec) {
                constexpr int ldw = DVc + 4, NG = DVc / 4;
                float* Ws = Ns;
                for (int idx = tid; idx < CC * NG; idx += kThreads) {
                    const int j = idx / NG, c = (idx % NG) * 4;
                    const float wj = j < L ? w(j) : 0.f;
                    const float* y = Y + j * ldv + c;
                    *reinterpret_cast<float4*>(Ws + j * ldw + c) =
                        make_float4(wj * y[0], wj * y[1], wj * y[2], wj * y[3]);
                }
                __syncthreads();
                for (int tI = tid; tI < DKc * NG / 4; tI += kThreads) {
                    const int d0 = (tI / NG) * 4, c0 = (tI % NG) * 4;
                    float u[4][4];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int e = 0; e < 4; ++e) u[r][e] = 0.f;
#pragma unroll 8
                    for (int j = 0; j < CC; ++j) {
                        const float4 wy = *reinterpret_cast<const float4*>(Ws + j * ldw + c0);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float x = X[j * ldk + d0 + r];
                            u[r][0] = fmaf(x, wy.x, u[r][0]);
                            u[r][1] = fmaf(x, wy.y, u[r][1]);
                            u[r][2] = fmaf(x, wy.z, u[r][2]);
                            u[r][3] = fmaf(x, wy.w, u[r][3]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float* sp = Ss + (d0 + r) * lds + c0 + e;
                            *sp = fmaf(gL, *sp, u[r][e]);
                        }
                }
            }
        };

        // A_ij = D_ij q~_i . k~_j (j <= i): tiles of 4 rows i and one column j
        for (int item = tid; item < (st_only ? 0 : ((L + 3) >> 2) * 32); item += kThreads) {
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
        // The forward sweep with the normaliser never forms n_i: with X_i = S dO_i and
        // B_ij = dO_i . v_j (j <= i), dO_i . n_i = sum_j A_ij B_ij + xi_i q~_i . X_i, and
        // the gradient's terms become P_ij = D_ij (B_ij / den_i + du_i) and
        // xi_i (X_i / den_i + du_i z), so the products with S and with V run once.
        const bool fwd_norm = role == 0 && !st_only && normalize;
        float* Xs = taylor ? TQ : Ns;  // X_i, rows ldk apart
        if (fwd_norm) {
            // B_ij into Ps (zero above the diagonal): tiles of 4 rows i and one column j
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
                    if (i < L && j < L) Ps[i * lda + j] = j <= i ? acc[r] : 0.f;
                }
            }
            // X_i = S dO_i
            tiles(L, dk, [&](int i0, int c0, int c1) {
                const int a0 = c0 < dk ? c0 : 0, a1 = c1 < dk ? c1 : 0;
                float it[4][2] = {};
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
                    if (c0 < dk) Xs[i * ldk + c0] = it[r][0];
                    if (c1 < dk) Xs[i * ldk + c1] = it[r][1];
                }
            });
            __syncthreads();
            // den_i, du_i (one warp per row: the sums over j, d_k)
            const int warp = tid >> 5, lane = tid & 31;
            for (int i = warp; i < L; i += kThreads / 32) {
                float r = 0.f, qz = 0.f, don = 0.f, qx = 0.f;
                for (int j = lane; j <= i; j += 32) {
                    const float a = As[i * lda + j];
                    r += a;
                    don = fmaf(a, Ps[i * lda + j], don);
                }
                for (int d = lane; d < dk; d += 32) {
                    const float q = Qs[i * ldk + d];
                    qz = fmaf(q, zs[d], qz);
                    qx = fmaf(q, Xs[i * ldk + d], qx);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    r += __shfl_xor_sync(0xffffffffu, r, off);
                    qz += __shfl_xor_sync(0xffffffffu, qz, off);
                    don += __shfl_xor_sync(0xffffffffu, don, off);
                    qx += __shfl_xor_sync(0xffffffffu, qx, off);
                }
                if (lane == 0) {
                    const float u = r + xi(i) * qz;
                    const float dd = norm_den(u, normalize, eps);
                    const float dd_du = normalize == 2 ? (fabsf(u) > 1.f ? (u > 0.f ? 1.f : -1.f) : 0.f)
                                                       : 1.f;
                    don = fmaf(xi(i), qx, don);  // dO_i . n_i
                    den[i] = dd;
                    du[i] = -don / (dd * dd) * dd_du;
                    stats[((size_t)bh * T_len + t0 + i) * 2] = dd;
                    stats[((size_t)bh * T_len + t0 + i) * 2 + 1] = du[i];
                }
            }
            __syncthreads();
            // P_ij = D_ij (B_ij / den_i + du_i), in place
            for (int idx = tid; idx < L * 32; idx += kThreads) {
                const int i = idx >> 5;
                for (int j = idx & 31; j < L; j += 32)
                    if (j <= i) Ps[i * lda + j] = (Ps[i * lda + j] / den[i] + du[i]) * dmask(i, j);
            }
            __syncthreads();
        }
        // dn_i = dO_i / den_i (in place; the backward sweep)
        if (normalize && need_qg && !fwd_norm) {
            for (int idx = tid; idx < L * dv; idx += kThreads) {
                const int i = idx / dv, cc2 = idx % dv;
                Gs[i * ldv + cc2] /= den[i];
            }
            __syncthreads();
        }
        // P_ij = D_ij (dn_i . v_j + du_i)  (j <= i): tiles of 4 rows i and one column j
        for (int item = tid; item < (st_only || fwd_norm ? 0 : ((L + 3) >> 2) * 32); item += kThreads) {
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
            // (with the normaliser S dn_i = X_i / den_i)
            if (!st_only) tiles(L, dk, [&](int i0, int c0, int c1) {
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
                for (int cc2 = 0; cc2 < (fwd_norm ? 0 : dv); ++cc2) {
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
                        float inter = fwd_norm ? Xs[i * ldk + d] / den[i] : it[r][e];
                        if (normalize) inter = fmaf(du[i], zs[d], inter);
                        float v = in[r][e] + xi(i) * inter;
                        if (phi) v *= fminf(1.f, Qs[i * ldk + d]);
                        if (taylor)
                            TQ[i * ldk + d] = v;
                        else
                            store_elem(dQ, qk_base + (size_t)(t0 + i) * dk + d, v);
                    }
                }
            });
            __syncthreads();
            // Taylor map: dq = the features' gradient through the map's transpose Jacobian
            if (taylor && !st_only) taylor_back(TQ, Qs, dQ, L, t0);
            // S = gamma^L S + sum_j zeta_j k~_j^T v_j ; z likewise
            if constexpr (kVec) {
                state_update(Ks, Vs, [&](int j) { return zt(j); }, gL);
            } else tiles(dk, dv, [&](int d0, int c0, int c1) {
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
                    if (d >= dk) continue;  // (dk need not be a multiple of 4)
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
            if (!st_only) tiles(L, dv, [&](int j0, int c0, int c1) {
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
            if (!st_only) tiles(L, dk, [&](int j0, int c0, int c1) {
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
                        if (taylor)
                            TQ[j * ldk + d] = v;
                        else
                            store_elem(dK, qk_base + (size_t)(t0 + j) * dk + d, v);
                    }
                }
            });
            __syncthreads();
            if (taylor && !st_only) taylor_back(TQ, Ks, dK, L, t0);  // dk through the map
            // G = gamma^L G + sum_i xi_i q~_i^T dn_i ;  Gz = gamma^L Gz + sum_i xi_i du_i q~_i
            if constexpr (kVec) {
                state_update(Qs, Gs, [&](int i) { return xi(i); }, gL);
            } else tiles(dk, dv, [&](int d0, int c0, int c1) {
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
                    if (d >= dk) continue;
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
    if (st_only) {  // this segment's own contribution (and its total log2 decay)
        float* agg = role == 0 ? sg.agg : sg.agg1;
        float* zagg = role == 0 ? sg.zagg : sg.zagg1;
        for (int idx = tid; idx < dk * dv; idx += kThreads)
            agg[sidx * dk * dv + idx] = Ss[(idx / dv) * lds + idx % dv];
        for (int d = tid; d < dk; d += kThreads) zagg[sidx * dk + d] = zs[d];
        if (role == 0 && log_a && sg.seg_l2 && tid == 0) sg.seg_l2[sidx] = seg_lam;
    } else if (role == 1 && seg == 0) {  // gradients of the initial state
        if (dS0)
            for (int idx = tid; idx < dk * dv; idx += kThreads)
                dS0[(size_t)bh * dk * dv + idx] = Ss[(idx / dv) * lds + idx % dv];
        if (dz0)
            for (int d = tid; d < dk; d += kThreads) dz0[(size_t)bh * dk + d] = zs[d];
    }
}

// Entry states of the segments from their own contributions (see the header).
// dir 0 (forward sweep): e(0) = init, e(q) = d(q-1) e(q-1) + agg(q-1);
// dir 1 (backward sweep): e(P-1) = init, e(q) = d(q+1) e(q+1) + agg(q+1);
// d(q) = gamma^len(q) (len(q) the tokens of segment q, the last one ragged) or
// 2^(seg_l2[bh][q]) with the per-token decay.  One thread per element of a
// sequence's state (d_k x d_v) and, with do_z, of z (d_k more); blockIdx.y
// picks the direction's arrays from `sc`.
struct ScanArgs {
    const float* init[2];
    const float* zinit[2];
    const float* agg[2];
    const float* zagg[2];
    float* ent[2];
    float* zent[2];
    int dir0;  // direction of blockIdx.y == 0
};

__global__ void bwd_scan_kernel(const __grid_constant__ ScanArgs sc, int BH, int H, int P, int seg_len,
                                int T, int dk, int dv, int do_z, const float* __restrict__ seg_l2,
                                const __grid_constant__ KernelGammas g) {
    const int dir = sc.dir0 + (int)blockIdx.y;
    const size_t per = (size_t)dk * dv + dk;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)BH * per) return;
    const size_t bh = idx / per;
    const size_t e = idx % per;
    const bool is_z = e >= (size_t)dk * dv;
    if (is_z && !do_z) return;
    const size_t n = is_z ? dk : (size_t)dk * dv;
    const size_t el = is_z ? e - (size_t)dk * dv : e;
    const float* init = is_z ? sc.zinit[blockIdx.y] : sc.init[blockIdx.y];
    const float* agg = is_z ? sc.zagg[blockIdx.y] : sc.agg[blockIdx.y];
    float* ent = is_z ? sc.zent[blockIdx.y] : sc.ent[blockIdx.y];
    const float l2g = g.log2g[bh % H];
    auto dec = [&](int q) {
        return seg_l2 ? exp2f(seg_l2[bh * P + q]) : gamma_pow(l2g, (float)min(seg_len, T - q * seg_len));
    };
    float x = init ? init[bh * n + el] : 0.f;
    for (int s = 0; s < P; ++s) {
        const int q = dir == 0 ? s : P - 1 - s;
        ent[(bh * P + q) * n + el] = x;
        // the next entry: segment q's decay and own contribution (forward: e(q+1);
        // backward: e(q-1))
        if (s + 1 < P) x = fmaf(dec(q), x, agg[(bh * P + q) * n + el]);
    }
}

// A segment's own contribution for the scan, as one weighted product over the
// segment's tokens s .. e-1: a contribution starts from zero, so the chunk
// recurrences above multiply out to one weight per token and no chunks are needed:
//   role 0: agg = sum_t w_t k~_t^T v_t,   zagg = sum_t w_t k~_t,
//           w_t = gamma^(e-1-t), or 2^(b_(e-1) - b_t) with the per-token decay;
//   role 1: agg = sum_t w_t q~_t^T dn_t,  zagg = sum_t w_t du_t q~_t,
//           w_t = gamma^(t-s+1), or 2^(b_t);
// b_t = sum_{u=s..t} log2 a_u, dn_t = do_t / den_t and du_t from the forward
// sweep's stats (dn = do, and no z, without the normaliser).  Role 0 also writes the
// segment's total log2 decay b_(e-1) with the per-token decay.
// 256 threads as a 16 x 16 grid: thread (ty, tx) holds rows ty DK/16 .. and columns
// tx DV/16 .. of the state.  The tokens pass through shared memory 32 at a time in
// fp32, double-buffered: the next tile's global loads are in flight while the
// current tile's products run.  A loader thread holds 8-element pieces of fixed
// columns, so it also sums its share of z; the shares are added in a fixed order.
constexpr int kGemmKT = 32;

template <int DK, int DV>
constexpr size_t gemm_smem_bytes() {
    return (size_t)2 * kGemmKT * (DK + DV) * sizeof(float);
}

template <typename T, int DK, int DV>
__global__ void __launch_bounds__(256) bwd_state_gemm_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    const T* __restrict__ dO, const float* __restrict__ stats, const float* __restrict__ log_a,
    int H, int T_len, int phi, int normalize, int role0, int seg_len,
    const __grid_constant__ KernelGammas g, const __grid_constant__ BwdSeg sg) {
    constexpr int KT = kGemmKT;
    constexpr int TM = DK / 16, TN = DV / 16;
    constexpr int GA = DK / 8, GB = DV / 8;      // 8-element pieces per row
    constexpr int RA = 256 / GA, RB = 256 / GB;  // rows per loader pass
    constexpr int NA = KT / RA, NB = KT / RB;    // loader passes per tile
    static_assert(TM % 4 == 0 && TN % 4 == 0 && NA >= 1 && NB >= 1, "shape");
    extern __shared__ __align__(16) float gsm[];
    float* As = gsm;                  // [2][KT][DK]
    float* Bs = gsm + 2 * KT * DK;    // [2][KT][DV]
    __shared__ float red[8];
    const float kLog2e = 1.44269504088896341f;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const int bh = blockIdx.x / sg.n_seg, seg = blockIdx.x % sg.n_seg;
    const size_t sidx = (size_t)bh * sg.n_seg + seg;
    const int role = role0 + (int)blockIdx.y;
    const int h = bh % H;
    const float l2g = g.log2g[h];
    const int s0 = seg * seg_len;
    const int e0 = min(T_len, s0 + seg_len);
    const int n_tiles = e0 > s0 ? (e0 - s0 + KT - 1) / KT : 0;
    const T* Ain = role == 0 ? K : Q;
    const T* Bin = role == 0 ? V : dO;
    const bool norm1 = role == 1 && normalize;
    const size_t tok0 = (size_t)bh * T_len;

    // the segment's total log2 decay (role 0, per-token decay)
    float total = 0.f;
    if (log_a && role == 0) {
        float acc = 0.f;
        for (int t = s0 + tid; t < e0; t += 256) acc += log_a[tok0 + t] * kLog2e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            float x = 0.f;
            for (int w = 0; w < 8; ++w) x += red[w];
            red[0] = x;
            if (sg.seg_l2) sg.seg_l2[sidx] = x;
        }
        __syncthreads();
        total = red[0];
    }

    const int pa = tid % GA, ra0 = tid / GA;
    const int pb = tid % GB, rb0 = tid / GB;
    Raw8<T> rawA[NA], rawB[NB];
    float lane_la = 0.f;                     // log2 a of token t0 + lane
    float2 lane_st = make_float2(1.f, 0.f);  // den, du of token t0 + lane
    float base = 0.f;                        // b up to the tile's first token (exclusive)
    float zacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto fetch = [&](int it) {
        const int t0 = s0 + it * KT;
#pragma unroll
        for (int n = 0; n < NA; ++n) {
            const int t = t0 + ra0 + RA * n;
            if (t < e0) rawA[n].load(Ain + (tok0 + t) * DK + pa * 8);
        }
#pragma unroll
        for (int n = 0; n < NB; ++n) {
            const int t = t0 + rb0 + RB * n;
            if (t < e0) rawB[n].load(Bin + (tok0 + t) * DV + pb * 8);
        }
        if (log_a) lane_la = t0 + lane < e0 ? log_a[tok0 + t0 + lane] * kLog2e : 0.f;
        if (norm1 && t0 + lane < e0) lane_st = *reinterpret_cast<const float2*>(stats + (tok0 + t0 + lane) * 2);
    };
    // the fetched tile, weighted, into buffer `buf`
    auto stage = [&](int it, int buf) {
        const int t0 = s0 + it * KT;
        float pre = 0.f;  // b of token t0 + lane (inclusive)
        if (log_a) {
            pre = lane_la;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o) pre += y;
            }
            pre += base;
            base = __shfl_sync(0xffffffffu, pre, 31);
        }
#pragma unroll
        for (int n = 0; n < NA; ++n) {
            const int r = ra0 + RA * n, t = t0 + r;
            float x[8];
            rawA[n].to_f32(x);
            float w;
            if (log_a) {
                const float br = __shfl_sync(0xffffffffu, pre, r);
                w = role == 0 ? exp2f(total - br) : exp2f(br);
            } else {
                w = gamma_pow(l2g, role == 0 ? (float)(e0 - 1 - t) : (float)(t - s0 + 1));
            }
            const float du = __shfl_sync(0xffffffffu, lane_st.y, r);
            const bool ok = t < e0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float v = x[j];
                if (phi) v = phi_elu1(v);
                v = ok ? v * w : 0.f;  // (past the end: the loads were skipped)
                x[j] = v;
                if (normalize) zacc[j] = fmaf(role == 0 ? 1.f : du, v, zacc[j]);
            }
            float4* dst = reinterpret_cast<float4*>(As + ((size_t)buf * KT + r) * DK + pa * 8);
            dst[0] = make_float4(x[0], x[1], x[2], x[3]);
            dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
#pragma unroll
        for (int n = 0; n < NB; ++n) {
            const int r = rb0 + RB * n, t = t0 + r;
            float y[8];
            rawB[n].to_f32(y);
            const float den = __shfl_sync(0xffffffffu, lane_st.x, r);
            const bool ok = t < e0;
#pragma unroll
            for (int j = 0; j < 8; ++j) y[j] = ok ? (norm1 ? y[j] / den : y[j]) : 0.f;
            float4* dst = reinterpret_cast<float4*>(Bs + ((size_t)buf * KT + r) * DV + pb * 8);
            dst[0] = make_float4(y[0], y[1], y[2], y[3]);
            dst[1] = make_float4(y[4], y[5], y[6], y[7]);
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n) acc[m][n] = 0.f;
    if (n_tiles > 0) {
        fetch(0);
        stage(0, 0);
    }
    __syncthreads();
    for (int it = 0; it < n_tiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < n_tiles) fetch(it + 1);
        const float* a_t = As + (size_t)buf * KT * DK + ty * TM;
        const float* b_t = Bs + (size_t)buf * KT * DV + tx * TN;
#pragma unroll 4
        for (int kk = 0; kk < KT; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int m = 0; m < TM; m += 4) {
                const float4 v = *reinterpret_cast<const float4*>(a_t + kk * DK + m);
                a[m] = v.x, a[m + 1] = v.y, a[m + 2] = v.z, a[m + 3] = v.w;
            }
#pragma unroll
            for (int n = 0; n < TN; n += 4) {
                const float4 v = *reinterpret_cast<const float4*>(b_t + kk * DV + n);
                b[n] = v.x, b[n + 1] = v.y, b[n + 2] = v.z, b[n + 3] = v.w;
            }
#pragma unroll
            for (int m = 0; m < TM; ++m)
#pragma unroll
                for (int n = 0; n < TN; ++n) acc[m][n] = fmaf(a[m], b[n], acc[m][n]);
        }
        if (it + 1 < n_tiles) stage(it + 1, buf ^ 1);
        __syncthreads();
    }
    float* agg = role == 0 ? sg.agg : sg.agg1;
    float* zagg = role == 0 ? sg.zagg : sg.zagg1;
#pragma unroll
    for (int m = 0; m < TM; ++m) {
        float* row = agg + (sidx * DK + ty * TM + m) * DV + tx * TN;
#pragma unroll
        for (int n = 0; n < TN; n += 4)
            *reinterpret_cast<float4*>(row + n) = make_float4(acc[m][n], acc[m][n + 1], acc[m][n + 2], acc[m][n + 3]);
    }
    // z: the loader threads' shares of each column, added row group by row group
    float* zpart = gsm;  // [RA][DK] (the tiles are no longer read)
#pragma unroll
    for (int j = 0; j < 8; ++j) zpart[ra0 * DK + pa * 8 + j] = zacc[j];
    __syncthreads();
    for (int d = tid; d < DK; d += 256) {
        float z = 0.f;
        for (int r = 0; r < RA; ++r) z += zpart[r * DK + d];
        zagg[sidx * DK + d] = z;
    }
}

}  // namespace

int bwd_chunk_len(int dk, int dv, bool taylor) {
    int C = 32;
    while (C > 8 && (size_t)bwd_layout(C, dk, dv, taylor).total * 4 > 227 * 1024) C >>= 1;
    return C;
}

namespace {

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// The backward pass's segment plan and workspace layout (byte offsets).
struct BwdPlan {
    int C, n_chunks, P, seg_chunks;
    size_t smem;
    size_t o_stats, o_a0, o_a0z, o_e0, o_e0z, o_a1, o_a1z, o_e1, o_e1z, o_l2, bytes;
};

// dk: the state's rows (1 + d + d^2 with the Taylor map)
BwdPlan bwd_plan(int B, int H, int T, int dk, int dv, bool normalize, bool taylor) {
    BwdPlan pl;
    pl.C = bwd_chunk_len(dk, dv, taylor);
    pl.smem = (size_t)bwd_layout(pl.C, dk, dv, taylor).total * sizeof(float);
    pl.n_chunks = T > 0 ? (T + pl.C - 1) / pl.C : 0;
    const size_t nbh = (size_t)B * H;
    // CTAs an SM holds by shared memory (registers allow four), and as many segments
    // per sequence as fill every SM that often, each of two chunks or more
    const int per_sm = (int)std::min<size_t>(4, std::max<size_t>(1, (227 * 1024) / pl.smem));
    size_t want = nbh ? ((size_t)device_sms() * per_sm) / nbh : 1;
    want = std::min<size_t>(want, (size_t)std::max(1, pl.n_chunks / 2));
    pl.P = (int)std::max<size_t>(1, want);
    pl.seg_chunks = pl.P > 1 ? (pl.n_chunks + pl.P - 1) / pl.P : std::max(1, pl.n_chunks);
    if (pl.P > 1) pl.P = (pl.n_chunks + pl.seg_chunks - 1) / pl.seg_chunks;  // segments used
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    pl.o_stats = normalize ? take(nbh * T * 2 * sizeof(float)) : 0;
    const size_t st = nbh * pl.P * dk * dv * sizeof(float), zt = nbh * pl.P * dk * sizeof(float);
    if (pl.P > 1) {
        pl.o_a0 = take(st), pl.o_a0z = take(zt), pl.o_e0 = take(st), pl.o_e0z = take(zt);
        pl.o_a1 = take(st), pl.o_a1z = take(zt), pl.o_e1 = take(st), pl.o_e1z = take(zt);
        pl.o_l2 = take(nbh * pl.P * sizeof(float));
    } else {
        pl.o_a0 = pl.o_a0z = pl.o_e0 = pl.o_e0z = pl.o_a1 = pl.o_a1z = pl.o_e1 = pl.o_e1z = pl.o_l2 = 0;
    }
    pl.bytes = off;
    return pl;
}

}  // namespace

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int bwd_state_rows(const BwdArgs& a) { return a.taylor ? taylor_feature_dim(a.dk) : a.dk; }

size_t bwd_stats_offset(const BwdArgs& a) {
    return a.T > 0 ? bwd_plan(a.B, a.H, a.T, bwd_state_rows(a), a.dv, a.normalize, a.taylor).o_stats : 0;
}

size_t bwd_workspace_bytes(const BwdArgs& a) {
    return a.T > 0 ? bwd_plan(a.B, a.H, a.T, bwd_state_rows(a), a.dv, a.normalize, a.taylor).bytes : 0;
}

cudaError_t launch_chunk_bwd_simt(const BwdArgs& a, const KernelGammas& g, cudaStream_t s) {
    const int ds = bwd_state_rows(a);  // the state's rows; a.dk is the width of Q and K
    const BwdPlan pl = bwd_plan(a.B, a.H, a.T, ds, a.dv, a.normalize, a.taylor);
    const int C = pl.C;
    const size_t smem = pl.smem;
    const unsigned nbh = (unsigned)((size_t)a.B * a.H);
    const int nm = norm_mode(a.normalize, a.floor_norm);
    char* ws = static_cast<char*>(a.workspace);
    float* stats = nm ? reinterpret_cast<float*>(ws + pl.o_stats) : nullptr;
    auto fp = [&](size_t o) { return reinterpret_cast<float*>(ws + o); };
    BwdSeg base;
    std::memset(&base, 0, sizeof(base));
    base.n_seg = pl.P;
    base.seg_chunks = pl.seg_chunks;
    BwdSeg full = base, st = base;
    if (pl.P > 1) {
        full.S_ent = fp(pl.o_e0), full.z_ent = fp(pl.o_e0z);
        full.G_ent = fp(pl.o_e1), full.Gz_ent = fp(pl.o_e1z);
        st.state_only = 1;
        st.agg = fp(pl.o_a0), st.zagg = fp(pl.o_a0z), st.agg1 = fp(pl.o_a1), st.zagg1 = fp(pl.o_a1z);
        st.seg_l2 = a.log_a ? fp(pl.o_l2) : nullptr;
    }
    cudaError_t e = cudaSuccess;
    auto launch = [&](auto kern, auto cast, int role0, unsigned roles, const BwdSeg& sg) {
        if (e != cudaSuccess) return;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return;
        TraceScope trace(sg.state_only ? "chunk_bwd_simt_kernel/state"
                         : roles == 2 ? "chunk_bwd_simt_kernel"
                         : role0 == 0 ? "chunk_bwd_simt_kernel/dq" : "chunk_bwd_simt_kernel/dkdv",
                         s);
        kern<<<dim3(nbh * pl.P, roles), kThreads, smem, s>>>(
            cast(a.Q), cast(a.K), cast(a.V), cast(a.dO), a.S0, a.z0, a.dS_T, a.dz_T, cast(a.dQ),
            cast(a.dK), cast(a.dV), a.dS0, a.dz0, stats, a.H, a.T, ds, a.dv, C, a.phi, nm,
            a.eps, role0, a.log_a, g, sg, a.dk, a.taylor ? 1 : 0);
        e = cudaGetLastError();
    };
    // the entry states of direction dir0 (and dir0 + 1 when dirs == 2)
    auto scan = [&](int dir0, int dirs) {
        if (e != cudaSuccess) return;
        ScanArgs sc;
        std::memset(&sc, 0, sizeof(sc));
        sc.dir0 = dir0;
        for (int y = 0; y < dirs; ++y) {
            const int dir = dir0 + y;
            sc.init[y] = dir == 0 ? a.S0 : a.dS_T;
            sc.zinit[y] = dir == 0 ? a.z0 : a.dz_T;
            sc.agg[y] = fp(dir == 0 ? pl.o_a0 : pl.o_a1);
            sc.zagg[y] = fp(dir == 0 ? pl.o_a0z : pl.o_a1z);
            sc.ent[y] = fp(dir == 0 ? pl.o_e0 : pl.o_e1);
            sc.zent[y] = fp(dir == 0 ? pl.o_e0z : pl.o_e1z);
        }
        const size_t total = (size_t)nbh * ((size_t)ds * a.dv + ds);
        TraceScope trace("bwd_scan_kernel", s);
        bwd_scan_kernel<<<dim3((unsigned)((total + 255) / 256), dirs), 256, 0, s>>>(
            sc, (int)nbh, a.H, pl.P, pl.seg_chunks * C, a.T, ds, a.dv, nm ? 1 : 0,
            a.log_a ? fp(pl.o_l2) : nullptr, g);
        e = cudaGetLastError();
    };
    // the segments' own contributions: the weighted product where its shape is
    // built, else a state-only pass of the chunked kernel
    const bool gemm_ok = !a.taylor && (a.dk == 64 || a.dk == 128) && (a.dv == 64 || a.dv == 128) &&
                         aligned16(a.Q) && aligned16(a.K) && aligned16(a.V) && aligned16(a.dO);
    auto contributions = [&](auto kern, auto cast, int role0, unsigned roles) {
        if (!gemm_ok) {
            launch(kern, cast, role0, roles, st);
            return;
        }
        if (e != cudaSuccess) return;
        auto go = [&](auto gk, size_t bytes) {
            e = cudaFuncSetAttribute(gk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e != cudaSuccess) return;
            TraceScope trace("bwd_state_gemm_kernel", s);
            gk<<<dim3(nbh * pl.P, roles), 256, bytes, s>>>(
                cast(a.Q), cast(a.K), cast(a.V), cast(a.dO), stats, a.log_a, a.H, a.T, a.phi, nm,
                role0, pl.seg_chunks * C, g, st);
            e = cudaGetLastError();
        };
        using E = std::remove_pointer_t<decltype(cast(a.Q))>;
        if (a.dk == 64 && a.dv == 64) go(bwd_state_gemm_kernel<E, 64, 64>, gemm_smem_bytes<64, 64>());
        else if (a.dk == 64) go(bwd_state_gemm_kernel<E, 64, 128>, gemm_smem_bytes<64, 128>());
        else if (a.dv == 64) go(bwd_state_gemm_kernel<E, 128, 64>, gemm_smem_bytes<128, 64>());
        else go(bwd_state_gemm_kernel<E, 128, 128>, gemm_smem_bytes<128, 128>());
    };
    auto run = [&](auto kern, auto cast) {
        if (a.dq_only) {  // the forward sweep alone
            if (pl.P > 1) {
                contributions(kern, cast, 0, 1);
                scan(0, 1);
            }
            launch(kern, cast, 0, 1, full);
            return;
        }
        if (pl.P <= 1) {
            if (nm == 0) {
                launch(kern, cast, 0, 2, full);  // the two sweeps are independent
            } else {
                launch(kern, cast, 0, 1, full);  // the backward sweep reads the forward sweep's den, du
                launch(kern, cast, 1, 1, full);
            }
            return;
        }
        if (nm == 0) {  // both sweeps' contributions, entries, then both sweeps
            contributions(kern, cast, 0, 2);
            scan(0, 2);
            launch(kern, cast, 0, 2, full);
        } else {  // the backward sweep's contributions need the forward sweep's den, du
            contributions(kern, cast, 0, 1);
            scan(0, 1);
            launch(kern, cast, 0, 1, full);
            contributions(kern, cast, 1, 1);
            scan(1, 1);
            launch(kern, cast, 1, 1, full);
        }
    };
    auto bf = [](const void* p) { return (__nv_bfloat16*)const_cast<void*>(p); };
    const bool plain = !a.taylor && C == 32 && gemm_ok;  // (gemm_ok: 16-byte aligned rows)
    if (a.bf16 && plain && a.dk == 64 && a.dv == 64)
        run(chunk_bwd_simt_kernel<__nv_bfloat16, 64, 64, 32>, bf);
    else if (a.bf16 && plain && a.dk == 128 && a.dv == 128)
        run(chunk_bwd_simt_kernel<__nv_bfloat16, 128, 128, 32>, bf);
    else if (a.bf16)
        run(chunk_bwd_simt_kernel<__nv_bfloat16>, bf);
    else
        run(chunk_bwd_simt_kernel<float>, [](const void* p) { return (float*)const_cast<void*>(p); });
    return e;
}

}  // namespace la
