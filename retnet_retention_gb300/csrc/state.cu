// State initialisation and copy kernels: the empty state S_0 = 0, z_0 = 0 of
// the recurrent form ("Linear attention", zerotofrontier 21.2, box "Causal
// linear attention, recurrent form"), and the S_T = S_0 hand-off of an empty
// sequence.  Plain bandwidth kernels: 16-byte stores, grid-stride loops.
#include "launch.h"
#include "trace.h"

namespace la {

__global__ void __launch_bounds__(256) state_zero_kernel(float4* S4, size_t n4, float* z,
                                                         size_t nz) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    for (size_t i = i0; i < n4; i += stride) S4[i] = zero;
    for (size_t i = i0; i < nz; i += stride) z[i] = 0.f;
}

__global__ void __launch_bounds__(256) state_copy_kernel(float4* dst, const float4* src,
                                                         size_t n4) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
        dst[i] = src[i];
}

static int grid_for(size_t work) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
    size_t blocks = (work + 255) / 256;
    size_t cap = (size_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

// n_S is a multiple of 16 floats (d_v is a multiple of 16), so float4 covers it.
cudaError_t launch_state_zero(float* S, float* z, size_t n_S, size_t n_z, cudaStream_t s) {
    if (n_S == 0 && n_z == 0) return cudaSuccess;
    size_t n4 = n_S / 4;
    TraceScope trace("state_zero_kernel", s);
    state_zero_kernel<<<grid_for(n4 > n_z ? n4 : n_z), 256, 0, s>>>(
        reinterpret_cast<float4*>(S), n4, z, z ? n_z : 0);
    return cudaGetLastError();
}

// n is a multiple of 4 floats (the state sizes are multiples of 16).
cudaError_t launch_state_copy(float* dst, const float* src, size_t n, cudaStream_t s) {
    if (n == 0 || dst == src) return cudaSuccess;
    size_t n4 = n / 4;
    TraceScope trace("state_copy_kernel", s);
    state_copy_kernel<<<grid_for(n4), 256, 0, s>>>(reinterpret_cast<float4*>(dst),
                                                   reinterpret_cast<const float4*>(src), n4);
    return cudaGetLastError();
}

}  // namespace la
