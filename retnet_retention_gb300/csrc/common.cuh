// Shared device/host helpers of liblinattn (the CUDA path only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/linattn.h"

namespace la {

// Largest head count a call may use: per-head decays travel in the kernel
// parameter block (see KernelGammas).
constexpr int kMaxHeads = 256;

// Per-head decay values in the kernel parameters: gamma itself (fp32, as the
// caller gave it) and log2(gamma) rounded from a double-precision log, used
// for powers gamma^n = exp2(n * log2 gamma) (exact 1 when gamma == 1).
struct KernelGammas {
    float gamma[kMaxHeads];
    float log2g[kMaxHeads];
};

__device__ __forceinline__ float load_elem(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// phi(x) = elu(x) + 1: x + 1 above zero, e^x at or below it.
// Normaliser denominator from d = phi(q)^T z: mode 1 adds eps, mode 2 floors
// |d| at 1 (LA_NORM_FLOOR).
__device__ __forceinline__ float norm_den(float d, int mode, float eps) {
    return mode == 2 ? fmaxf(fabsf(d), 1.f) : d + eps;
}

__device__ __forceinline__ float phi_elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }

// gamma^n for n >= 0 from the host-rounded log2(gamma).
__device__ __forceinline__ float gamma_pow(float log2g, float n) { return exp2f(n * log2g); }

}  // namespace la
