// Backward pass on the tensor cores, by running the chunkwise forward three
// times with the roles of its inputs exchanged.
//
// The gradients of o_t = q_t S_t, S_t = gamma S_{t-1} + k_t^T v_t (no feature
// map, no normaliser) for L = sum_t do_t . o_t + <dS_T, S_T> are
//
//   dq_t = sum_{s<=t} gamma^(t-s) (do_t . v_s) k_s + gamma^(t+1) do_t S_0^T
//        = the forward pass with queries dO, keys V, values K, initial state S_0^T;
//   G_t  = q_t^T do_t + gamma G_{t+1} (G = dL/dS_t, G_{T-1} includes dS_T),
//   dv_t = k_t G_t,   dk_t = G_t v_t:
//        in reversed time t' = T-1-t, G is a forward state with keys q and values
//        dO, so dV is the forward pass over the reversed sequences with queries K,
//        keys Q, values dO, and dK the one with queries V, keys dO, values Q; both
//        start from dS_T / gamma (dS_T enters G_{T-1} undecayed, while the forward
//        pass decays its initial state once before the first token), and
//        dS_0 = gamma G_0 is gamma times the dV pass's final state.
//
// "Linear attention" (zerotofrontier 21.2), "Decoding, training, and what each
// costs": the gradients are cumulative sums, forward in time for the queries and
// backward in time for the keys and values.  The reversed copies cost one read
// and one write of Q, K, V and dO and of the two reversed outputs; where the
// pipelined kernel's factored build applies (every gamma in (0, 1] with
// gamma^(C-1) >= 2^-64) it walks the sequences backward itself instead, on the
// original tensors.
//
// With phi = elu + 1 (no normaliser) the passes run on phi(q), phi(k), and the q and
// k gradients go through phi'(x) (1 above zero, e^x at or below) at the end.
//
// Normalised calls (d_v = 64) split: dq and the per-token denominators from the
// CUDA-core kernel's forward sweep, dk and dv from two reversed-time passes over
// augmented operands (the section "The normalised backward" below).
#include <algorithm>
#include <cstring>

#include "launch.h"
#include "trace.h"

namespace la {

namespace {

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// phi = elu + 1 of two bf16 tensors of n8 x 8 elements: a~ = bf16(phi(a)), b~ likewise
// (8 elements an item).
__global__ void __launch_bounds__(256) phi_prep_kernel(const __nv_bfloat16* __restrict__ a,
                                                       const __nv_bfloat16* __restrict__ b,
                                                       __nv_bfloat16* __restrict__ at,
                                                       __nv_bfloat16* __restrict__ bt, size_t n8) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n8;
         i += (size_t)gridDim.x * blockDim.x) {
        const bool second = i >= n8;
        const size_t j = second ? i - n8 : i;
        const uint4 u = reinterpret_cast<const uint4*>(second ? b : a)[j];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[e] = pack2(phi_elu1(__uint_as_float(w[e] << 16)), phi_elu1(__uint_as_float(w[e] & 0xffff0000u)));
        reinterpret_cast<uint4*>(second ? bt : at)[j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Gradients through phi for two tensors of n8 x 8 elements: out = bf16(g phi'(x)),
// phi'(x) = 1 above zero, e^x at or below (8 elements an item).
__global__ void __launch_bounds__(256) phi_grad_pair_kernel(
    const __nv_bfloat16* __restrict__ ga, const __nv_bfloat16* __restrict__ xa, __nv_bfloat16* __restrict__ oa,
    const __nv_bfloat16* __restrict__ gb, const __nv_bfloat16* __restrict__ xb, __nv_bfloat16* __restrict__ ob,
    size_t n8) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n8;
         i += (size_t)gridDim.x * blockDim.x) {
        const bool second = i >= n8;
        const size_t j = second ? i - n8 : i;
        const uint4 g = reinterpret_cast<const uint4*>(second ? gb : ga)[j];
        const uint4 x = reinterpret_cast<const uint4*>(second ? xb : xa)[j];
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, xw[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(xw[e] << 16), x1 = __uint_as_float(xw[e] & 0xffff0000u);
            o[e] = pack2(__uint_as_float(gw[e] << 16) * (x0 > 0.f ? 1.f : expf(x0)),
                         __uint_as_float(gw[e] & 0xffff0000u) * (x1 > 0.f ? 1.f : expf(x1)));
        }
        reinterpret_cast<uint4*>(second ? ob : oa)[j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// out[bh][t][:] = in[bh][T-1-t][:] for a [BH][T][d] bf16 tensor (16-byte pieces).
__global__ void __launch_bounds__(256) reverse_time_kernel(const uint4* __restrict__ in,
                                                           uint4* __restrict__ out, int T,
                                                           int pieces_per_row, size_t total) {
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t row = idx / pieces_per_row;
        const int p = (int)(idx % pieces_per_row);
        const size_t bh = row / T;
        const int t = (int)(row % T);
        out[idx] = in[(bh * T + (T - 1 - t)) * pieces_per_row + p];
    }
}

// out[bh][j][i] = scale[h] * in[bh][i][j] (transpose = 1) or scale[h] * in[bh][i][j].
__global__ void __launch_bounds__(256) state_scale_kernel(const float* __restrict__ in,
                                                          float* __restrict__ out, int H, int R,
                                                          int Cc, int transpose, int inverse,
                                                          const __grid_constant__ KernelGammas g) {
    const size_t per = (size_t)R * Cc;
    const size_t total = per * gridDim.y;
    const size_t bh = blockIdx.y;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per;
         e += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(e / Cc), j = (int)(e % Cc);
        const float gm = g.gamma[bh % H];
        const float s = inverse ? 1.f / gm : gm;
        const float x = in[bh * per + e] * s;
        if (transpose) out[bh * per + (size_t)j * R + i] = x;
        else out[bh * per + e] = x;
    }
    (void)total;
}

// out[b][j][i] = scale[h] * in[b][i][j] for b < nb matrices of R x Cc (R, Cc multiples
// of 32; the input's matrices in_per elements apart, its first R rows read),
// through 32 x 32 tiles in shared memory so that both the reads and the writes take
// whole rows.  Block (32, 8); grid (Cc / 32, R / 32, nb).
__global__ void __launch_bounds__(256) state_transpose_kernel(const float* __restrict__ in,
                                                              float* __restrict__ out, int H, int R,
                                                              int Cc, size_t in_per, int inverse,
                                                              const __grid_constant__ KernelGammas g) {
    __shared__ float tile[32][33];
    const size_t b = blockIdx.z;
    const size_t per = (size_t)R * Cc;  // (input matrices are in_per apart)
    const float gm = g.gamma[b % H];
    const float sc = inverse ? 1.f / gm : gm;
    const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
    for (int r = threadIdx.y; r < 32; r += 8)
        tile[r][threadIdx.x] = in[b * in_per + (size_t)(i0 + r) * Cc + j0 + threadIdx.x];
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8)
        out[b * per + (size_t)(j0 + r) * R + i0 + threadIdx.x] = sc * tile[threadIdx.x][r];
}

cudaError_t reverse_time(const void* in, void* out, size_t nbh, int T, int d, cudaStream_t s) {
    const int ppr = d * 2 / 16;
    const size_t total = nbh * (size_t)T * ppr;
    const unsigned blocks = (unsigned)std::min<size_t>((total + 255) / 256, 152 * 16);
    TraceScope trace("reverse_time_kernel", s);
    reverse_time_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(in),
                                               static_cast<uint4*>(out), T, ppr, total);
    return cudaGetLastError();
}

cudaError_t state_scale(const float* in, float* out, size_t nbh, int H, int R, int Cc,
                        bool transpose, bool inverse, const KernelGammas& g, cudaStream_t s) {
    if (transpose && R % 32 == 0 && Cc % 32 == 0 && nbh <= 65535) {
        TraceScope trace("state_transpose_kernel", s);
        state_transpose_kernel<<<dim3((unsigned)(Cc / 32), (unsigned)(R / 32), (unsigned)nbh), dim3(32, 8),
                                 0, s>>>(in, out, H, R, Cc, (size_t)R * Cc, inverse ? 1 : 0, g);
        return cudaGetLastError();
    }
    const size_t per = (size_t)R * Cc;
    dim3 grid((unsigned)std::min<size_t>((per + 255) / 256, 64), (unsigned)nbh);
    TraceScope trace("state_scale_kernel", s);
    state_scale_kernel<<<grid, 256, 0, s>>>(in, out, H, R, Cc, transpose ? 1 : 0, inverse ? 1 : 0, g);
    return cudaGetLastError();
}

// A forward call's arguments: bf16, causal, no flags.
ChunkArgs fwd_args(const void* Q, const void* K, const void* V, void* O, const float* S0,
                   float* S_out, int B, int H, int T, int dk, int dv, void* ws, size_t ws_bytes,
                   int* dev_status) {
    ChunkArgs c;
    std::memset(&c, 0, sizeof(c));
    c.Q = Q; c.K = K; c.V = V; c.O = O; c.S0 = S0; c.S_out = S_out;
    c.B = B; c.H = H; c.T = T; c.dk = dk; c.dv = dv;
    c.bf16 = true;
    c.workspace = ws;
    c.workspace_bytes = ws_bytes;
    c.dev_status = dev_status;
    return c;
}

// Workspace layout: reversed Q, K, V, dO, reversed dV, dK outputs, the states,
// the dV pass's segment contributions and their transposes, then the forward
// calls' own workspace (one call at a time).
struct BwdTcPlan {
    size_t o_qr, o_kr, o_vr, o_dor, o_dvr, o_dkr, o_s0t, o_g0, o_g0t, o_gfin, o_agg, o_aggt, o_qt,
        o_kt, o_dqt, o_dkt, o_fwd, fwd_bytes, bytes;
    // the dV and dK passes have the same segments (more than one): the dK pass's
    // state walk is the dV pass's transposed (keys dO and values Q instead of keys
    // Q and values dO), so it is not run again
    bool share;
    int n_seg;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

BwdTcPlan bwd_tc_plan(const BwdArgs& a) {
    BwdTcPlan p;
    const size_t nbh = (size_t)a.B * a.H;
    const size_t nqk = align256(nbh * a.T * a.dk * 2), nv = align256(nbh * a.T * a.dv * 2);
    const size_t ns = align256(nbh * a.dk * a.dv * 4);
    size_t off = 0;
    p.o_qr = off; off += nqk;
    p.o_kr = off; off += nqk;
    p.o_vr = off; off += nv;
    p.o_dor = off; off += nv;
    p.o_dvr = off; off += nv;
    p.o_dkr = off; off += nqk;
    p.o_s0t = off; off += ns;
    p.o_g0 = off; off += ns;
    p.o_g0t = off; off += ns;
    p.o_gfin = off; off += ns;
    const ChunkArgs c1 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dv, a.dk, nullptr, 0, nullptr);
    const ChunkArgs c2 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dk, a.dv, nullptr, 0, nullptr);
    int n2 = 1, sc2 = 0, n3 = 1, sc3 = 0;
    tc_segments(c2, &n2, &sc2);
    tc_segments(c1, &n3, &sc3);  // (the dK pass has the dQ pass's shape)
    p.share = n2 > 1 && n2 == n3 && sc2 == sc3;
    p.n_seg = n2;
    const size_t nagg = p.share ? align256(nbh * n2 * a.dk * a.dv * 4) : 0;
    p.o_agg = off; off += nagg;
    p.o_aggt = off; off += nagg;
    // with phi: phi(q), phi(k) and the gradients before phi'
    const size_t nphi = a.phi ? nqk : 0;
    p.o_qt = off; off += nphi;
    p.o_kt = off; off += nphi;
    p.o_dqt = off; off += nphi;
    p.o_dkt = off; off += nphi;
    p.o_fwd = off;
    p.fwd_bytes = std::max(tc_workspace_bytes(c1), tc_workspace_bytes(c2));
    p.bytes = off + p.fwd_bytes;
    return p;
}

// ---- The normalised backward (phi or not, floored or not): dq on the CUDA cores,
// dk and dv on the tensor cores.
//
// With n_t = q~_t S_t, u_t = q~_t . z_t, dd_t = max(|u_t|, 1) or u_t + eps and
// o_t = n_t / dd_t, the loss's gradients with respect to n_t and u_t are
// dn_t = do_t / dd_t and du_t = -(do_t . o_t) / dd_t * dd'(u_t), and
//   dq~_t = S_t dn_t + du_t z_t,
//   dk~_t = G_t v_t + Gz_t = sum_{s>=t} gamma^(s-t) (v_t . dn_s + du_s) q~_s (+ the
//           final-state terms),   dv_t = k~_t G_t
// ("Linear attention" page, "Decoding, training, and what each costs": the gradients
// are cumulative sums; the normalised form of "Transformers are RNNs", section 3.2).
// dq~ is a near-cancellation (dn_t . (v_s - o_t) summed against positive k~_s): bf16
// operands put it at 1-3.5e-2 of its largest element (fp64 emulations of the kernel's
// roundings on short windows), so dq and the per-token dd, du come from the CUDA-core
// kernel's forward sweep in fp32.  dk and dv keep 2-3x inside the bf16 tolerance as
// reversed-time forward passes with augmented operands: dk~ with queries
// [v | 1 | 1], keys [dn | du_hi | du_lo] (du split into two bf16 parts, so that the
// sum keeps about 16 bits), values q~; dv with queries k~, keys q~, values dn.  The
// augmented operands are stored 72 wide and read as 128 by the d_k = 128 build (the
// tensor maps fill the columns past the row with zeros); dn is read in place as the
// first 64 columns of [dn | du]; the dv pass takes its segments' contributions from
// the dk~ pass's (the transpose of their first 64 rows).  d_v = 64.

constexpr int kAugW = 128;   // width of the augmented operands in the kernel
constexpr int kAugCols = 72; // ... as stored (64 value columns, du_hi and du_lo or two ones, 6 zeros)

// Per token row: q~ = phi(q), k~ = phi(k) and the augmented [dn | du_hi | du_lo | 0]
// and [v | 1 | 1 | 0] (kAugCols wide, dn = do / dd in bf16).  One thread per 16-byte
// piece of a row (pieces 0..7 carry the 64 value columns, piece 8 the two extra
// columns and zeros; pieces below d_k / 8 carry q~ and k~).
__global__ void __launch_bounds__(256) aug_prep_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
    const __nv_bfloat16* __restrict__ V, const __nv_bfloat16* __restrict__ dO,
    const float* __restrict__ stats, __nv_bfloat16* __restrict__ qt, __nv_bfloat16* __restrict__ kt,
    __nv_bfloat16* __restrict__ xq, __nv_bfloat16* __restrict__ xk, size_t rows, int dk, int phi) {
    constexpr int dv = 64;
    const int pieces = max(kAugCols / 8, dk / 8);
    const size_t total = rows * pieces;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t row = idx / pieces;
        const int pc = (int)(idx % pieces);
        uint4 wq = make_uint4(0u, 0u, 0u, 0u), wk = make_uint4(0u, 0u, 0u, 0u);
        if (pc < dv / 8) {
            const float inv = 1.f / stats[row * 2];
            const uint4 g = *reinterpret_cast<const uint4*>(dO + row * dv + pc * 8);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack2(__uint_as_float(gw[e] << 16) * inv, __uint_as_float(gw[e] & 0xffff0000u) * inv);
            wq = make_uint4(o[0], o[1], o[2], o[3]);
            wk = *reinterpret_cast<const uint4*>(V + row * dv + pc * 8);
        } else if (pc == dv / 8) {
            const float du = stats[row * 2 + 1];
            const __nv_bfloat16 hi = __float2bfloat16_rn(du);
            const __nv_bfloat16 lo = __float2bfloat16_rn(du - __bfloat162float(hi));
            wq.x = (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
            wk.x = 0x3F803F80u;  // two bf16 ones
        }
        if (pc < kAugCols / 8) {
            *reinterpret_cast<uint4*>(xq + row * kAugCols + pc * 8) = wq;
            *reinterpret_cast<uint4*>(xk + row * kAugCols + pc * 8) = wk;
        }
        if (pc < dk / 8) {
            const uint4 a = *reinterpret_cast<const uint4*>(Q + row * dk + pc * 8);
            const uint4 b = *reinterpret_cast<const uint4*>(K + row * dk + pc * 8);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
            uint32_t oq[4], ok[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q0 = __uint_as_float(aw[e] << 16), q1 = __uint_as_float(aw[e] & 0xffff0000u);
                float k0 = __uint_as_float(bw[e] << 16), k1 = __uint_as_float(bw[e] & 0xffff0000u);
                if (phi) {
                    q0 = phi_elu1(q0), q1 = phi_elu1(q1), k0 = phi_elu1(k0), k1 = phi_elu1(k1);
                }
                oq[e] = pack2(q0, q1);
                ok[e] = pack2(k0, k1);
            }
            *reinterpret_cast<uint4*>(qt + row * dk + pc * 8) = make_uint4(oq[0], oq[1], oq[2], oq[3]);
            *reinterpret_cast<uint4*>(kt + row * dk + pc * 8) = make_uint4(ok[0], ok[1], ok[2], ok[3]);
        }
    }
}

// The dk~ pass's initial state [b][128][d_k] from dS_T [b][d_k][d_v] (null: zero) and
// dz_T [b][d_k] (null: zero), over gamma_h: rows 0 .. d_v-1 hold dS_T's transpose,
// row d_v dz_T (the queries' two ones read the sum of rows d_v and d_v + 1), the
// rest zeros.
__global__ void __launch_bounds__(256) aug_state_kernel(const float* __restrict__ S,
                                                        const float* __restrict__ z,
                                                        float* __restrict__ out, size_t nbh, int H,
                                                        int dk, int dv,
                                                        const __grid_constant__ KernelGammas g) {
    const size_t total = nbh * kAugW * dk;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t b = e / ((size_t)kAugW * dk);
        const int c = (int)((e / dk) % kAugW), d = (int)(e % dk);
        float x = 0.f;
        if (c < dv && S) x = S[(b * dk + d) * dv + c];
        else if (c == dv && z) x = z[b * dk + d];
        out[e] = x / g.gamma[b % H];
    }
}

// The last step, one launch: dk = bf16(dk~ phi'(k)) 8 elements an item (phi'(x) = 1
// above zero, e^x at or below; 1 without phi), then dS_0 = gamma_h G_0 (the dv pass's
// final state, if wanted) and dz_0 = gamma_h (fin[b][d_v][d] + fin[b][d_v + 1][d])
// (the dk~ pass's final-state rows of du_hi and du_lo, if wanted), one element an item.
struct AugFinish {
    const __nv_bfloat16* gk;  // dk~
    const __nv_bfloat16* k;
    __nv_bfloat16* out_k;     // dk
    const float* gfin;        // [b][d_k][d_v] or null
    float* dS0;
    const float* gkfin;       // [b][128][d_k] or null
    float* dz0;
    size_t n8, nS, nz;
    int H, dk, dv, phi;
};

__global__ void __launch_bounds__(256) aug_finish_kernel(const __grid_constant__ AugFinish f,
                                                         const __grid_constant__ KernelGammas g) {
    const size_t total = f.n8 + f.nS + f.nz;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        if (i < f.n8) {
            const uint4 a = reinterpret_cast<const uint4*>(f.gk)[i];
            const uint4 b = reinterpret_cast<const uint4*>(f.k)[i];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float g0 = __uint_as_float(aw[e] << 16), g1 = __uint_as_float(aw[e] & 0xffff0000u);
                if (f.phi) {
                    const float x0 = __uint_as_float(bw[e] << 16), x1 = __uint_as_float(bw[e] & 0xffff0000u);
                    g0 *= x0 > 0.f ? 1.f : expf(x0);
                    g1 *= x1 > 0.f ? 1.f : expf(x1);
                }
                o[e] = pack2(g0, g1);
            }
            reinterpret_cast<uint4*>(f.out_k)[i] = make_uint4(o[0], o[1], o[2], o[3]);
        } else if (i < f.n8 + f.nS) {
            const size_t j = i - f.n8;
            const size_t b = j / ((size_t)f.dk * f.dv);
            f.dS0[j] = g.gamma[b % f.H] * f.gfin[j];
        } else {
            const size_t j = i - f.n8 - f.nS;
            const size_t b = j / f.dk;
            const int d = (int)(j % f.dk);
            const float* r = f.gkfin + b * kAugW * f.dk;
            f.dz0[j] = g.gamma[b % f.H] * (r[(size_t)f.dv * f.dk + d] + r[(size_t)(f.dv + 1) * f.dk + d]);
        }
    }
}

// The hybrid's workspace (byte offsets): the CUDA-core kernel's own (its per-token
// dd, du at offset bwd_stats_offset), then the tensor-core passes' operands and
// states, then the passes' own workspace.
struct BwdAugPlan {
    size_t o_qt, o_kt, o_xq, o_xk, o_dkt, o_gk0, o_g0, o_gkfin, o_gfin, o_aggk, o_aggv, o_fwd,
        fwd_bytes, bytes;
    // the dk~ and dv passes cut the sequences into the same segments (more than one):
    // the dv pass takes its contributions from the dk~ pass's state walk
    bool share;
    int n_seg;
};

ChunkArgs aug_pass_args(const BwdArgs& a, int width_qk, int width_v) {
    ChunkArgs c = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H, a.T,
                           width_qk, width_v, nullptr, 0, nullptr);
    c.reverse = true;
    return c;
}

bool aug_shape_ok(const BwdArgs& a) {
    if (!a.bf16 || !a.normalize || a.taylor || a.log_a || a.T <= 0 || opt_tc_lockstep()) return false;
    if (a.dv != 64 || (a.dk != 64 && a.dk != 128)) return false;
    return tc_supported(aug_pass_args(a, kAugW, a.dk)) && tc_supported(aug_pass_args(a, a.dk, a.dv));
}

BwdAugPlan bwd_aug_plan(const BwdArgs& a) {
    BwdAugPlan p;
    const size_t nbh = (size_t)a.B * a.H, rows = nbh * a.T;
    size_t off = align256(bwd_workspace_bytes(a));
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    p.o_qt = take(rows * a.dk * 2);
    p.o_kt = take(rows * a.dk * 2);
    p.o_xq = take(rows * kAugCols * 2);
    p.o_xk = take(rows * kAugCols * 2);
    p.o_dkt = take(rows * a.dk * 2);
    p.o_gk0 = take(nbh * kAugW * a.dk * sizeof(float));
    p.o_g0 = take(nbh * a.dk * a.dv * sizeof(float));
    p.o_gkfin = take(nbh * kAugW * a.dk * sizeof(float));
    p.o_gfin = take(nbh * a.dk * a.dv * sizeof(float));
    int nk = 1, sk = 0, nv = 1, sv = 0;
    tc_segments(aug_pass_args(a, kAugW, a.dk), &nk, &sk);
    tc_segments(aug_pass_args(a, a.dk, a.dv), &nv, &sv);
    p.share = nk > 1 && nk == nv && sk == sv;
    p.n_seg = nk;
    p.o_aggk = take(p.share ? nbh * nk * kAugW * a.dk * sizeof(float) : 0);
    p.o_aggv = take(p.share ? nbh * nk * a.dk * a.dv * sizeof(float) : 0);
    p.o_fwd = off;
    p.fwd_bytes = std::max(tc_workspace_bytes(aug_pass_args(a, kAugW, a.dk)),
                           tc_workspace_bytes(aug_pass_args(a, a.dk, a.dv)));
    p.bytes = off + p.fwd_bytes;
    return p;
}

unsigned grid_for(size_t work) {
    return (unsigned)std::max<size_t>(1, std::min<size_t>((work + 255) / 256, 152 * 16));
}

cudaError_t launch_aug(const BwdArgs& a, const KernelGammas& g, cudaStream_t s) {
    const BwdAugPlan p = bwd_aug_plan(a);
    if (!a.workspace || a.workspace_bytes < p.bytes) return cudaErrorInvalidValue;
    char* ws = static_cast<char*>(a.workspace);
    auto bp = [&](size_t o) { return reinterpret_cast<__nv_bfloat16*>(ws + o); };
    auto fp = [&](size_t o) { return reinterpret_cast<float*>(ws + o); };
    const size_t nbh = (size_t)a.B * a.H, rows = nbh * a.T;
    void* fws = ws + p.o_fwd;
    cudaError_t e = cudaSuccess;
    int launches = 0;
    // 1. the forward sweep on the CUDA cores: dq and the per-token dd, du
    BwdArgs a0 = a;
    a0.dq_only = true;
    a0.dK = a0.dV = nullptr;
    a0.dS0 = a0.dz0 = nullptr;
    if ((e = launch_chunk_bwd_simt(a0, g, s)) != cudaSuccess) return e;
    const float* stats = fp(bwd_stats_offset(a));
    // 2. the passes' operands
    __nv_bfloat16 *qt = bp(p.o_qt), *kt = bp(p.o_kt), *xq = bp(p.o_xq), *xk = bp(p.o_xk), *dkt = bp(p.o_dkt);
    {
        TraceScope trace("aug_prep_kernel", s);
        aug_prep_kernel<<<grid_for(rows * std::max(kAugCols / 8, a.dk / 8)), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a.Q), static_cast<const __nv_bfloat16*>(a.K),
            static_cast<const __nv_bfloat16*>(a.V), static_cast<const __nv_bfloat16*>(a.dO), stats,
            qt, kt, xq, xk, rows, a.dk, a.phi ? 1 : 0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 3. initial states of the reversed passes, entering after the last token:
    //    [dS_T^T; dz_T; 0] / gamma and dS_T / gamma
    float* gk0 = nullptr;
    float* g0 = nullptr;
    if (a.dS_T || a.dz_T) {
        gk0 = fp(p.o_gk0);
        TraceScope trace("aug_state_kernel", s);
        aug_state_kernel<<<grid_for(nbh * kAugW * a.dk), 256, 0, s>>>(a.dS_T, a.dz_T, gk0, nbh, a.H,
                                                                    a.dk, a.dv, g);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.dS_T) {
        g0 = fp(p.o_g0);
        if ((e = state_scale(a.dS_T, g0, nbh, a.H, a.dk, a.dv, false, true, g, s)) != cudaSuccess) return e;
    }
    // 4. dk~ in reversed time: queries [v | 1], keys [dn | du], values q~
    float* gkfin = a.dz0 ? fp(p.o_gkfin) : nullptr;
    ChunkArgs ck = aug_pass_args(a, kAugW, a.dk);
    ck.Q = xk; ck.K = xq; ck.V = qt; ck.O = dkt; ck.S0 = gk0; ck.S_out = gkfin;
    ck.qk_cols = ck.qk_pitch = kAugCols;
    ck.workspace = fws; ck.workspace_bytes = p.fwd_bytes;
    if (p.share) ck.agg = fp(p.o_aggk);
    if ((e = launch_chunk_tc(ck, g, s, &launches)) != cudaSuccess) return e;
    // 5. dv in reversed time: queries k~, keys q~, values dn; its final state is G_0
    float* gfin = a.dS0 ? fp(p.o_gfin) : nullptr;
    ChunkArgs cv = aug_pass_args(a, a.dk, a.dv);
    cv.Q = kt; cv.K = qt; cv.V = xq; cv.O = a.dV; cv.S0 = g0; cv.S_out = gfin;
    cv.v_pitch = kAugCols;  // dn: the first 64 columns of [dn | du]
    cv.workspace = fws; cv.workspace_bytes = p.fwd_bytes;
    if (p.share) {  // keys q~ with values dn give the transpose of keys dn with values q~
        cv.agg = fp(p.o_aggv);
        cv.agg_ready = true;
        KernelGammas one;
        std::memset(&one, 0, sizeof(one));
        for (int h = 0; h < kMaxHeads; ++h) one.gamma[h] = 1.f;
        TraceScope trace("state_transpose_kernel", s);
        state_transpose_kernel<<<dim3((unsigned)(a.dk / 32), (unsigned)(a.dv / 32), (unsigned)(nbh * p.n_seg)),
                                 dim3(32, 8), 0, s>>>(ck.agg, cv.agg, a.H, a.dv, a.dk,
                                                      (size_t)kAugW * a.dk, 0, one);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_chunk_tc(cv, g, s, &launches)) != cudaSuccess) return e;
    // 6. through phi (dk = dk~ phi'(k)) and the initial state's gradients
    //    (dS_0 = gamma G_0, dz_0 = gamma Gz_0), one launch
    AugFinish f;
    f.gk = dkt;
    f.k = static_cast<const __nv_bfloat16*>(a.K);
    f.out_k = static_cast<__nv_bfloat16*>(a.dK);
    f.gfin = gfin; f.dS0 = a.dS0; f.gkfin = gkfin; f.dz0 = a.dz0;
    f.n8 = rows * a.dk / 8;
    f.nS = a.dS0 ? nbh * a.dk * a.dv : 0;
    f.nz = a.dz0 ? nbh * a.dk : 0;
    f.H = a.H; f.dk = a.dk; f.dv = a.dv; f.phi = a.phi ? 1 : 0;
    TraceScope trace("aug_finish_kernel", s);
    aug_finish_kernel<<<grid_for(f.n8 + f.nS + f.nz), 256, 0, s>>>(f, g);
    return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
    if (a.normalize) return aug_shape_ok(a);
    if (!a.bf16 || a.taylor || a.log_a || a.T <= 0) return false;
    if ((a.dk != 64 && a.dk != 128) || (a.dv != 64 && a.dv != 128)) return false;
    const ChunkArgs c1 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dv, a.dk, nullptr, 0, nullptr);
    const ChunkArgs c2 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dk, a.dv, nullptr, 0, nullptr);
    return tc_supported(c1) && tc_supported(c2);
}

size_t bwd_tc_workspace_bytes(const BwdArgs& a) {
    // (normalised: the plan starts with the CUDA-core kernel's own workspace, which
    // also covers that kernel alone where a gamma rules out the reversed passes)
    if (a.normalize) return bwd_aug_plan(a).bytes;
    return bwd_tc_plan(a).bytes;
}

cudaError_t launch_chunk_bwd_tc(const BwdArgs& a, const KernelGammas& g, cudaStream_t s) {
    if (a.normalize) {
        ChunkArgs ck = aug_pass_args(a, kAugW, a.dk), cv = aug_pass_args(a, a.dk, a.dv);
        if (!tc_reverse_supported(ck, g) || !tc_reverse_supported(cv, g)) return launch_chunk_bwd_simt(a, g, s);
        return launch_aug(a, g, s);
    }
    const BwdTcPlan p = bwd_tc_plan(a);
    if (!a.workspace || a.workspace_bytes < p.bytes) return cudaErrorInvalidValue;
    char* ws = static_cast<char*>(a.workspace);
    const size_t nbh = (size_t)a.B * a.H;
    void* fws = ws + p.o_fwd;
    cudaError_t e = cudaSuccess;
    int launches = 0;
    // with phi = elu + 1 (no normaliser) the passes run on phi(q), phi(k) and their
    // gradients go through phi' at the end
    const void* Qp = a.Q;
    const void* Kp = a.K;
    void* dQp = a.dQ;
    void* dKp = a.dK;
    const size_t n8 = nbh * a.T * a.dk / 8;
    if (a.phi) {
        __nv_bfloat16* qt = reinterpret_cast<__nv_bfloat16*>(ws + p.o_qt);
        __nv_bfloat16* kt = reinterpret_cast<__nv_bfloat16*>(ws + p.o_kt);
        TraceScope trace("phi_prep_kernel", s);
        phi_prep_kernel<<<(unsigned)std::max<size_t>(1, std::min<size_t>((2 * n8 + 255) / 256, 152 * 16)), 256,
                          0, s>>>(static_cast<const __nv_bfloat16*>(a.Q),
                                  static_cast<const __nv_bfloat16*>(a.K), qt, kt, n8);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        Qp = qt;
        Kp = kt;
        dQp = ws + p.o_dqt;
        dKp = ws + p.o_dkt;
    }
    // dQ: queries dO, keys V, values K, initial state S_0^T
    float* s0t = nullptr;
    if (a.S0) {
        s0t = reinterpret_cast<float*>(ws + p.o_s0t);
        KernelGammas one;  // a plain transpose (scale 1)
        std::memset(&one, 0, sizeof(one));
        for (int h = 0; h < kMaxHeads; ++h) one.gamma[h] = 1.f;
        if ((e = state_scale(a.S0, s0t, nbh, a.H, a.dk, a.dv, true, false, one, s)) != cudaSuccess)
            return e;
    }
    ChunkArgs c1 = fwd_args(a.dO, a.V, Kp, dQp, s0t, nullptr, a.B, a.H, a.T, a.dv, a.dk, fws,
                            p.fwd_bytes, nullptr);
    if ((e = launch_chunk_tc(c1, g, s, &launches)) != cudaSuccess) return e;
    // initial states of the reversed passes: dS_T / gamma and its transpose
    float* g0 = nullptr;
    float* g0t = nullptr;
    if (a.dS_T) {
        g0 = reinterpret_cast<float*>(ws + p.o_g0);
        g0t = reinterpret_cast<float*>(ws + p.o_g0t);
        if ((e = state_scale(a.dS_T, g0, nbh, a.H, a.dk, a.dv, false, true, g, s)) != cudaSuccess)
            return e;
        if ((e = state_scale(a.dS_T, g0t, nbh, a.H, a.dk, a.dv, true, true, g, s)) != cudaSuccess)
            return e;
    }
    float* gfin = a.dS0 ? reinterpret_cast<float*>(ws + p.o_gfin) : nullptr;
    // dV: queries K, keys Q, values dO in reversed time, its final state G_0;
    // dK: queries V, keys dO, values Q in reversed time
    ChunkArgs c2 = fwd_args(Kp, Qp, a.dO, a.dV, g0, gfin, a.B, a.H, a.T, a.dk, a.dv, fws,
                            p.fwd_bytes, nullptr);
    ChunkArgs c3 = fwd_args(a.V, a.dO, Qp, dKp, g0t, nullptr, a.B, a.H, a.T, a.dv, a.dk, fws,
                            p.fwd_bytes, nullptr);
    c2.reverse = c3.reverse = true;
    if (tc_reverse_supported(c2, g) && tc_reverse_supported(c3, g)) {
        // the kernel walks the sequences backward itself: no copies
        if (p.share) {
            c2.agg = reinterpret_cast<float*>(ws + p.o_agg);
            c3.agg = reinterpret_cast<float*>(ws + p.o_aggt);
            c3.agg_ready = true;
        }
        if ((e = launch_chunk_tc(c2, g, s, &launches)) != cudaSuccess) return e;
        if (p.share) {  // the dK pass's contributions: sum dO^T Q = (sum Q^T dO)^T
            KernelGammas one;
            std::memset(&one, 0, sizeof(one));
            for (int h = 0; h < kMaxHeads; ++h) one.gamma[h] = 1.f;
            if ((e = state_scale(c2.agg, c3.agg, nbh * p.n_seg, a.H, a.dk, a.dv, true, false, one, s)) !=
                cudaSuccess)
                return e;
        }
        if ((e = launch_chunk_tc(c3, g, s, &launches)) != cudaSuccess) return e;
    } else {
        // reversed copies of the sequences, forward passes over them, the outputs
        // reversed back
        void* qr = ws + p.o_qr;
        void* kr = ws + p.o_kr;
        void* vr = ws + p.o_vr;
        void* dor = ws + p.o_dor;
        void* dvr = ws + p.o_dvr;
        void* dkr = ws + p.o_dkr;
        if ((e = reverse_time(Qp, qr, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
        if ((e = reverse_time(Kp, kr, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
        if ((e = reverse_time(a.V, vr, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        if ((e = reverse_time(a.dO, dor, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        c2.Q = kr; c2.K = qr; c2.V = dor; c2.O = dvr;
        c3.Q = vr; c3.K = dor; c3.V = qr; c3.O = dkr;
        c2.reverse = c3.reverse = false;
        if ((e = launch_chunk_tc(c2, g, s, &launches)) != cudaSuccess) return e;
        if ((e = launch_chunk_tc(c3, g, s, &launches)) != cudaSuccess) return e;
        if ((e = reverse_time(dvr, a.dV, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        if ((e = reverse_time(dkr, dKp, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
    }
    if (a.dS0) {  // dS_0 = gamma G_0
        if ((e = state_scale(gfin, a.dS0, nbh, a.H, a.dk, a.dv, false, false, g, s)) != cudaSuccess)
            return e;
    }
    if (a.phi) {  // dq = dq~ phi'(q), dk = dk~ phi'(k)
        TraceScope trace("phi_grad_pair_kernel", s);
        phi_grad_pair_kernel<<<(unsigned)std::max<size_t>(1, std::min<size_t>((2 * n8 + 255) / 256, 152 * 16)),
                               256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(dQp), static_cast<const __nv_bfloat16*>(a.Q),
            static_cast<__nv_bfloat16*>(a.dQ), static_cast<const __nv_bfloat16*>(dKp),
            static_cast<const __nv_bfloat16*>(a.K), static_cast<__nv_bfloat16*>(a.dK), n8);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace la
