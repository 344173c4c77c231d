// Recurrent decode step (one token for every (b, h)), state updated in place:
//
//   S = gamma S + phi(k) v^T ;  z = gamma z + phi(k) ;  o = phi(q)^T S [/ (phi(q)^T z + eps)]
//
// "RetNet" (bembew), "Recurrent Representation"; "Linear attention"
// (zerotofrontier 21.2), the decode step: update first, then read.  With a
// per-token decay, gamma is this step's a = e^(log a) of the (b, h) ("Linear
// Attention, RWKV, and RetNet" 13.3, subsection 4: the gated decay G_t).
//
// The step is bound by HBM: every call reads and writes the whole fp32 state
// (d_k * d_v * 8 bytes per head) and does 4 d_k d_v flops per head.  One CTA
// owns one (b, h) state block.  Each thread owns 4 consecutive value columns
// (a float4) of a set of rows, so a warp reads whole 512-byte row segments;
// rows are streamed in batches of 16 float4 loads per thread that are issued
// before any of them is used (the first batch even before q, k, v are read),
// keeping up to 64 KB per CTA in flight.  The
// read-out sum over d_k is a register accumulation followed by a shared-
// memory reduction across the row slots.
//
// With the Taylor feature map ("Linear attention", "A Taylor feature map") q
// and k are 16 wide and the state has 1 + 16 + 256 = 273 rows in the page's
// order: phi(x) = (1, x, vec(x x^T)/sqrt 2) is built in shared memory first.
#include "launch.h"
#include "trace.h"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 16;
constexpr int kMaxRows = 288;  // feature rows held in shared memory (273 with the Taylor map)

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) decode_step_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    T* __restrict__ o, float* __restrict__ S, float* __restrict__ z, int H, int dk, int dv,
    int phi, int normalize, float eps, const float* __restrict__ log_a, int taylor,
    const __grid_constant__ KernelGammas g) {
    __shared__ float qf[kMaxRows];
    __shared__ float kf[kMaxRows];
    __shared__ float qk_in[32];
    __shared__ float red[kThreads * 4];
    __shared__ float den_part[kThreads / 32];

    const int bh = blockIdx.x;
    const int h = bh % H;
    const int din = dk;                           // width of q and k
    if (taylor) dk = 1 + din + din * din;         // rows of the state
    const float gam = log_a ? exp2f(log_a[bh] * 1.44269504088896341f) : g.gamma[h];
    const int tid = threadIdx.x;
    const int tpr = dv >> 2;           // threads per state row
    const int rpi = kThreads / tpr;    // rows per pass over the block
    const int cg = tid % tpr;          // my float4 column group
    const int rs = tid / tpr;          // my first row
    const int row4 = dv >> 2;          // float4 per row
    float4* Sb = reinterpret_cast<float4*>(S + (size_t)bh * dk * dv);

    // The state block is the only large read: issue the first batch of its
    // loads before anything else so their latency overlaps the q/k/v loads.
    float4 s[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        int i = rs + u * rpi;
        if (i < dk) s[u] = __ldcs(Sb + (size_t)i * row4 + cg);
    }
    if (taylor) {
        if (tid < 2 * din) qk_in[tid] = load_elem(tid < din ? q : k, (size_t)bh * din + tid % din);
        __syncthreads();
        for (int f = tid; f < dk; f += kThreads) {  // (1, x, x_a x_b / sqrt 2 row-major)
            float a = 1.f, b = 1.f;
            if (f >= 1 && f <= din) {
                a = qk_in[f - 1];
                b = qk_in[din + f - 1];
            } else if (f > din) {
                const int i = (f - 1 - din) / din, j = (f - 1 - din) % din;
                a = qk_in[i] * qk_in[j] * 0.70710678118654752f;
                b = qk_in[din + i] * qk_in[din + j] * 0.70710678118654752f;
            }
            qf[f] = a;
            kf[f] = b;
        }
    } else if (tid < dk) {
        float qv = load_elem(q, (size_t)bh * dk + tid);
        float kv = load_elem(k, (size_t)bh * dk + tid);
        qf[tid] = phi ? phi_elu1(qv) : qv;
        kf[tid] = phi ? phi_elu1(kv) : kv;
    }
    float vv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) vv[c] = load_elem(v, (size_t)bh * dv + cg * 4 + c);
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i0 = rs;; ) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            int i = i0 + u * rpi;
            if (i < dk) {
                const float kk = kf[i], qq = qf[i];
                float4 x = s[u];
                x.x = fmaf(gam, x.x, kk * vv[0]);
                x.y = fmaf(gam, x.y, kk * vv[1]);
                x.z = fmaf(gam, x.z, kk * vv[2]);
                x.w = fmaf(gam, x.w, kk * vv[3]);
                __stcs(Sb + (size_t)i * row4 + cg, x);
                acc[0] = fmaf(qq, x.x, acc[0]);
                acc[1] = fmaf(qq, x.y, acc[1]);
                acc[2] = fmaf(qq, x.z, acc[2]);
                acc[3] = fmaf(qq, x.w, acc[3]);
            }
        }
        i0 += rpi * kBatch;
        if (i0 >= dk) break;
        // next batch (only when d_k * d_v > 1024 * kBatch)
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            int i = i0 + u * rpi;
            if (i < dk) s[u] = __ldcs(Sb + (size_t)i * row4 + cg);
        }
    }
    // red[rs][col] for the rpi row slots
#pragma unroll
    for (int c = 0; c < 4; ++c) red[rs * dv + cg * 4 + c] = acc[c];

    float den = 1.f;
    if (normalize) {
        float part = 0.f;
        for (int f = tid; f < dk; f += kThreads) {
            float* zb = z + (size_t)bh * dk;
            float zi = fmaf(gam, zb[f], kf[f]);
            zb[f] = zi;
            part += qf[f] * zi;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if ((tid & 31) == 0) den_part[tid >> 5] = part;
    }
    __syncthreads();
    if (normalize) {
        float d = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) d += den_part[w];
        den = norm_den(d, normalize, eps);
    }
    for (int j = tid; j < dv; j += kThreads) {
        float sum = 0.f;
        for (int r = 0; r < rpi; ++r) sum += red[r * dv + j];
        store_elem(o, (size_t)bh * dv + j, normalize ? sum / den : sum);
    }
}

}  // namespace

cudaError_t launch_decode_step(const StepArgs& a, const KernelGammas& g, cudaStream_t s) {
    const size_t nbh = (size_t)a.B * a.H;
    if (nbh == 0) return cudaSuccess;
    if (nbh > 0x7fffffffu) return cudaErrorInvalidValue;
    dim3 grid((unsigned)nbh);
    TraceScope trace("decode_step_kernel", s);
    if (a.bf16) {
        decode_step_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
            (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
            (__nv_bfloat16*)a.o, a.S, a.z, a.H, a.dk, a.dv, a.phi, norm_mode(a.normalize, a.floor_norm), a.eps,
            a.log_a, a.taylor ? 1 : 0, g);
    } else {
        decode_step_kernel<float><<<grid, kThreads, 0, s>>>(
            (const float*)a.q, (const float*)a.k, (const float*)a.v, (float*)a.o, a.S, a.z,
            a.H, a.dk, a.dv, a.phi, norm_mode(a.normalize, a.floor_norm), a.eps, a.log_a,
            a.taylor ? 1 : 0, g);
    }
    return cudaGetLastError();
}

}  // namespace la
