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
#include <algorithm>
#include <cstring>

#include "launch.h"
#include "trace.h"

namespace la {

namespace {

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
// of 32), through 32 x 32 tiles in shared memory so that both the reads and the
// writes take whole rows.  Block (32, 8); grid (Cc / 32, R / 32, nb).
__global__ void __launch_bounds__(256) state_transpose_kernel(const float* __restrict__ in,
                                                              float* __restrict__ out, int H, int R,
                                                              int Cc, int inverse,
                                                              const __grid_constant__ KernelGammas g) {
    __shared__ float tile[32][33];
    const size_t b = blockIdx.z;
    const size_t per = (size_t)R * Cc;
    const float gm = g.gamma[b % H];
    const float sc = inverse ? 1.f / gm : gm;
    const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
    for (int r = threadIdx.y; r < 32; r += 8)
        tile[r][threadIdx.x] = in[b * per + (size_t)(i0 + r) * Cc + j0 + threadIdx.x];
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
                                 0, s>>>(in, out, H, R, Cc, inverse ? 1 : 0, g);
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
    size_t o_qr, o_kr, o_vr, o_dor, o_dvr, o_dkr, o_s0t, o_g0, o_g0t, o_gfin, o_agg, o_aggt, o_fwd,
        fwd_bytes, bytes;
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
    p.o_fwd = off;
    p.fwd_bytes = std::max(tc_workspace_bytes(c1), tc_workspace_bytes(c2));
    p.bytes = off + p.fwd_bytes;
    return p;
}

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
    if (!a.bf16 || a.phi || a.taylor || a.normalize || a.log_a || a.T <= 0) return false;
    if ((a.dk != 64 && a.dk != 128) || (a.dv != 64 && a.dv != 128)) return false;
    const ChunkArgs c1 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dv, a.dk, nullptr, 0, nullptr);
    const ChunkArgs c2 = fwd_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, a.B, a.H,
                                  a.T, a.dk, a.dv, nullptr, 0, nullptr);
    return tc_supported(c1) && tc_supported(c2);
}

size_t bwd_tc_workspace_bytes(const BwdArgs& a) { return bwd_tc_plan(a).bytes; }

cudaError_t launch_chunk_bwd_tc(const BwdArgs& a, const KernelGammas& g, cudaStream_t s) {
    const BwdTcPlan p = bwd_tc_plan(a);
    if (!a.workspace || a.workspace_bytes < p.bytes) return cudaErrorInvalidValue;
    char* ws = static_cast<char*>(a.workspace);
    const size_t nbh = (size_t)a.B * a.H;
    void* fws = ws + p.o_fwd;
    cudaError_t e = cudaSuccess;
    int launches = 0;
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
    ChunkArgs c1 = fwd_args(a.dO, a.V, a.K, a.dQ, s0t, nullptr, a.B, a.H, a.T, a.dv, a.dk, fws,
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
    ChunkArgs c2 = fwd_args(a.K, a.Q, a.dO, a.dV, g0, gfin, a.B, a.H, a.T, a.dk, a.dv, fws,
                            p.fwd_bytes, nullptr);
    ChunkArgs c3 = fwd_args(a.V, a.dO, a.Q, a.dK, g0t, nullptr, a.B, a.H, a.T, a.dv, a.dk, fws,
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
        if ((e = reverse_time(a.Q, qr, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
        if ((e = reverse_time(a.K, kr, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
        if ((e = reverse_time(a.V, vr, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        if ((e = reverse_time(a.dO, dor, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        c2.Q = kr; c2.K = qr; c2.V = dor; c2.O = dvr;
        c3.Q = vr; c3.K = dor; c3.V = qr; c3.O = dkr;
        c2.reverse = c3.reverse = false;
        if ((e = launch_chunk_tc(c2, g, s, &launches)) != cudaSuccess) return e;
        if ((e = launch_chunk_tc(c3, g, s, &launches)) != cudaSuccess) return e;
        if ((e = reverse_time(dvr, a.dV, nbh, a.T, a.dv, s)) != cudaSuccess) return e;
        if ((e = reverse_time(dkr, a.dK, nbh, a.T, a.dk, s)) != cudaSuccess) return e;
    }
    if (a.dS0) {  // dS_0 = gamma G_0
        if ((e = state_scale(gfin, a.dS0, nbh, a.H, a.dk, a.dv, false, false, g, s)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace la
