// Chunkwise forward on the CUDA cores in fp32 (the exact-fp32 path, and the
// path for any shape the tensor-core kernel does not take).
//
// "Chunked Recurrent Representation" ("RetNet", bembew): the sequence is cut
// into chunks of C tokens; inside a chunk the parallel form, across chunks
// the carried state.  The pages give the chunkwise form only in words; the
// equations, written out from the recurrence S_t = gamma S_{t-1} + k_t v_t^T,
// for a chunk of L <= C rows with local indices i, j and entry state S_{c-1}:
//
//   A_ij = (phi(q_i) . phi(k_j)) gamma^(i-j)  for j <= i, else 0
//   o_i  = sum_j A_ij v_j + gamma^(i+1) phi(q_i)^T S_{c-1}
//   den_i = sum_j A_ij + gamma^(i+1) phi(q_i)^T z_{c-1}            (normalising)
//   S_c  = gamma^L S_{c-1} + sum_j gamma^(L-1-j) phi(k_j) v_j^T
//   z_c  = gamma^L z_{c-1} + sum_j gamma^(L-1-j) phi(k_j)
//
// Only non-negative powers of gamma appear, so small gamma underflows to 0
// instead of overflowing.  With a per-token decay a_t (log a_t given) the
// powers become cumulative log-decays inside the chunk, b_i = sum_{s<=i} log a_s:
// gamma^(i-j) -> e^(b_i - b_j), gamma^(i+1) -> e^(b_i), gamma^(L-1-j) ->
// e^(b_(L-1) - b_j), gamma^L -> e^(b_(L-1)) (exponents again never positive).  The non-causal form (gamma = 1, "Linear
// attention" box) is two passes: the summary S = sum_t phi(k_t) v_t^T, then
// o_t = phi(q_t)^T S.
//
// One CTA owns one (b, h) and a block of up to 64 value columns and walks the
// chunks in order; S (d_k x 64 fp32) stays in shared memory for the whole
// sequence.  Inputs are read once per column block.
#include "launch.h"
#include "trace.h"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxDvBlock = 64;

struct SimtSmem {
    // offsets (in floats) into dynamic shared memory
    int q, k, v, a, s, z, den, pw, cum, xw, total;
};

__host__ __device__ inline SimtSmem simt_layout(int C, int dk, int dvb) {
    SimtSmem L;
    const int ld = dk + 1;  // odd row stride: column walks hit distinct banks
    L.q = 0;
    L.k = L.q + C * ld;
    L.v = L.k + C * ld;
    L.a = L.v + C * dvb;
    L.s = L.a + C * (C + 1);
    L.z = L.s + dk * dvb;
    L.den = L.z + dk;
    L.pw = L.den + C;
    L.cum = L.pw + C + 2;
    L.xw = L.cum + C;
    L.total = L.xw + C;
    return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
    T* __restrict__ O, const float* __restrict__ S0, const float* __restrict__ z0,
    float* __restrict__ S_out, float* __restrict__ z_out, int H, int T_len, int dk, int dv,
    int C, int dvb, int phi, int normalize, int noncausal, float eps,
    const float* __restrict__ log_a, const __grid_constant__ KernelGammas g) {
    extern __shared__ float smem[];
    const SimtSmem lay = simt_layout(C, dk, dvb);
    float* Qs = smem + lay.q;
    float* Ks = smem + lay.k;
    float* Vs = smem + lay.v;
    float* As = smem + lay.a;
    float* Ss = smem + lay.s;
    float* zs = smem + lay.z;
    float* den = smem + lay.den;
    float* pw = smem + lay.pw;
    float* cum = smem + lay.cum;  // per-token decay: log2 of the cumulative decay in the chunk
    float* xw = smem + lay.xw;    // per-token decay: e^(b_i) (pw then holds e^(b_(L-1) - b_j))
    const int ld = dk + 1;
    const int lda = C + 1;

    const int bh = blockIdx.x;
    const int h = bh % H;
    const int v0 = blockIdx.y * dvb;
    const int nv = min(dvb, dv - v0);
    const int tid = threadIdx.x;
    const float l2g = g.log2g[h];

    // gamma^n, n = 0..C
    for (int n = tid; n <= C; n += kThreads) pw[n] = gamma_pow(l2g, (float)n);
    // entry state
    for (int idx = tid; idx < dk * dvb; idx += kThreads) {
        int d = idx / dvb, c = idx % dvb;
        Ss[idx] = (S0 && c < nv) ? S0[((size_t)bh * dk + d) * dv + v0 + c] : 0.f;
    }
    for (int d = tid; d < dk; d += kThreads) zs[d] = z0 ? z0[(size_t)bh * dk + d] : 0.f;
    __syncthreads();

    const size_t qk_base = (size_t)bh * T_len * dk;
    const size_t v_base = (size_t)bh * T_len * dv;
    const int n_chunks = (T_len + C - 1) / C;
    // non-causal: pass 0 builds the summary, pass 1 reads it
    const int passes = noncausal ? 2 : 1;
    for (int pass = 0; pass < passes; ++pass) {
        const bool do_state = !noncausal || pass == 0;
        const bool do_out = !noncausal || pass == 1;
        for (int c = 0; c < n_chunks; ++c) {
            const int t0 = c * C;
            const int L = min(C, T_len - t0);
            // stage phi(Q_c), phi(K_c), V_c block in fp32
            for (int idx = tid; idx < L * dk; idx += kThreads) {
                int i = idx / dk, d = idx % dk;
                size_t gi = qk_base + (size_t)(t0 + i) * dk + d;
                if (do_out) {
                    float x = load_elem(Q, gi);
                    Qs[i * ld + d] = phi ? phi_elu1(x) : x;
                }
                float y = load_elem(K, gi);
                Ks[i * ld + d] = phi ? phi_elu1(y) : y;
            }
            for (int idx = tid; idx < L * dvb; idx += kThreads) {
                int i = idx / dvb, cc = idx % dvb;
                Vs[idx] = cc < nv ? load_elem(V, v_base + (size_t)(t0 + i) * dv + v0 + cc) : 0.f;
            }
            if (log_a && tid == 0) {  // b_i = sum_{s<=i} log a_s, in log2 units
                float acc = 0.f;
                for (int i = 0; i < L; ++i) {
                    acc += log_a[(size_t)bh * T_len + t0 + i] * 1.44269504088896341f;
                    cum[i] = acc;
                }
            }
            __syncthreads();
            if (log_a) {
                for (int i = tid; i < L; i += kThreads) {
                    xw[i] = exp2f(cum[i]);
                    pw[i] = exp2f(cum[L - 1] - cum[i]);
                }
                __syncthreads();
            }
            // decay factors of this chunk (see the header)
            auto dmask = [&](int i, int j) { return log_a ? exp2f(cum[i] - cum[j]) : pw[i - j]; };
            auto xi = [&](int i) { return log_a ? xw[i] : pw[i + 1]; };
            auto zeta = [&](int j) { return log_a ? pw[j] : pw[L - 1 - j]; };

            if (do_out) {
                if (!noncausal) {
                    // intra-chunk scores with the decay mask
                    for (int idx = tid; idx < L * L; idx += kThreads) {
                        int i = idx / L, j = idx % L;
                        float a = 0.f;
                        if (j <= i) {
                            const float* qi = Qs + i * ld;
                            const float* kj = Ks + j * ld;
                            float dot = 0.f;
                            for (int d = 0; d < dk; ++d) dot = fmaf(qi[d], kj[d], dot);
                            a = dot * dmask(i, j);
                        }
                        As[i * lda + j] = a;
                    }
                    __syncthreads();
                }
                if (normalize) {
                    for (int i = tid; i < L; i += kThreads) {
                        float r = 0.f;
                        if (!noncausal)
                            for (int j = 0; j <= i; ++j) r += As[i * lda + j];
                        float qz = 0.f;
                        for (int d = 0; d < dk; ++d) qz = fmaf(Qs[i * ld + d], zs[d], qz);
                        den[i] = norm_den(r + (noncausal ? 1.f : xi(i)) * qz, normalize, eps);
                    }
                    __syncthreads();
                }
                for (int idx = tid; idx < L * nv; idx += kThreads) {
                    int i = idx / nv, cc = idx % nv;
                    float intra = 0.f;
                    if (!noncausal)
                        for (int j = 0; j <= i; ++j) intra = fmaf(As[i * lda + j], Vs[j * dvb + cc], intra);
                    float inter = 0.f;
                    const float* qi = Qs + i * ld;
                    for (int d = 0; d < dk; ++d) inter = fmaf(qi[d], Ss[d * dvb + cc], inter);
                    float o = intra + (noncausal ? 1.f : xi(i)) * inter;
                    if (normalize) o = o / den[i];
                    store_elem(O, v_base + (size_t)(t0 + i) * dv + v0 + cc, o);
                }
                __syncthreads();
            }
            if (do_state) {
                // S_c = gamma^L S_{c-1} + sum_j gamma^(L-1-j) phi(k_j) v_j^T
                const float gL = noncausal ? 1.f : (log_a ? exp2f(cum[L - 1]) : pw[L]);
                for (int idx = tid; idx < dk * dvb; idx += kThreads) {
                    int d = idx / dvb, cc = idx % dvb;
                    float u = 0.f;
                    for (int j = 0; j < L; ++j) {
                        float w = noncausal ? 1.f : zeta(j);
                        u = fmaf(w * Ks[j * ld + d], Vs[j * dvb + cc], u);
                    }
                    Ss[idx] = fmaf(gL, Ss[idx], u);
                }
                for (int d = tid; d < dk; d += kThreads) {
                    float u = 0.f;
                    for (int j = 0; j < L; ++j) u = fmaf(noncausal ? 1.f : zeta(j), Ks[j * ld + d], u);
                    zs[d] = fmaf(gL, zs[d], u);
                }
                __syncthreads();
            }
        }
    }
    if (S_out) {
        for (int idx = tid; idx < dk * nv; idx += kThreads) {
            int d = idx / nv, cc = idx % nv;
            S_out[((size_t)bh * dk + d) * dv + v0 + cc] = Ss[d * dvb + cc];
        }
    }
    if (z_out && blockIdx.y == 0)
        for (int d = tid; d < dk; d += kThreads) z_out[(size_t)bh * dk + d] = zs[d];
}

}  // namespace

static int simt_dvb(int dv) { return dv < kMaxDvBlock ? dv : kMaxDvBlock; }

int simt_chunk_len(int requested, int dk) {
    int C = requested > 0 ? requested : 32;
    // shrink until the tile fits the 227 KB shared-memory limit
    while (C > 16 && (size_t)simt_layout(C, dk, kMaxDvBlock).total * 4 > 227 * 1024) C >>= 1;
    return C;
}

cudaError_t launch_chunk_simt(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s) {
    const int C = simt_chunk_len(a.chunk, a.dk);
    const int dvb = simt_dvb(a.dv);
    const size_t smem = (size_t)simt_layout(C, a.dk, dvb).total * sizeof(float);
    dim3 grid((unsigned)((size_t)a.B * a.H), (a.dv + dvb - 1) / dvb);
    cudaError_t e;
    TraceScope trace("chunk_simt_kernel", s);
    if (a.bf16) {
        auto kern = chunk_simt_kernel<__nv_bfloat16>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, s>>>(
            (const __nv_bfloat16*)a.Q, (const __nv_bfloat16*)a.K, (const __nv_bfloat16*)a.V,
            (__nv_bfloat16*)a.O, a.S0, a.z0, a.S_out, a.z_out, a.H, a.T,
            a.dk, a.dv, C, dvb, a.phi, norm_mode(a.normalize, a.floor_norm), a.noncausal, a.eps,
            a.log_a, g);
    } else {
        auto kern = chunk_simt_kernel<float>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreads, smem, s>>>(
            (const float*)a.Q, (const float*)a.K, (const float*)a.V, (float*)a.O, a.S0,
            a.z0, a.S_out, a.z_out, a.H, a.T, a.dk, a.dv, C, dvb, a.phi,
            norm_mode(a.normalize, a.floor_norm), a.noncausal, a.eps, a.log_a, g);
    }
    return cudaGetLastError();
}

}  // namespace la
