// la_chunk_fwd_noalloc: the chunkwise forward for callers that cannot
// allocate device memory.
//
// la_chunk_fwd needs caller-provided scratch (the per-segment states of a
// long sequence split across SMs).  Some callers cannot call cudaMalloc or
// hold no device allocator of their own: a plugin inside a host framework
// that owns every device allocation and hands the plugin only its inputs
// and outputs, or a serving loop that must not allocate once it is running
// (cudaMalloc can synchronise the device and can fail under memory
// pressure).  For them this entry point takes its scratch from one fixed,
// file-scope device array instead.  It allocates nothing itself.
//
// The array is la_noalloc_scratch below (LA_NOALLOC_SCRATCH_BYTES, 16 MiB).
// Every GPU that loads this library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current and caches it.
#include <cstdint>
#include <mutex>

#include "launch.h"

static __device__ __align__(256) unsigned char la_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr with *err set.
void* scratch_address(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, la_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" {

la_status la_chunk_fwd_noalloc(const void* Q, const void* K, const void* V, la_dtype dtype,
                               const float* gamma, int B, int H, int T, int d_k, int d_v,
                               unsigned flags, float eps, const float* S0, const float* z0,
                               void* O, float* S_out, float* z_out, int chunk, int* dev_status,
                               la_stream_t stream) {
    const size_t need = la_workspace_size(B, H, T, d_k, d_v, dtype, flags, chunk);
    if (need > (size_t)LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_INVALID_ARG;
    void* ws = nullptr;
    if (need > 0) {
        cudaError_t e = cudaSuccess;
        ws = scratch_address(&e);
        if (!ws) return LA_ERR_CUDA;
    }
    return la_chunk_fwd(Q, K, V, dtype, gamma, B, H, T, d_k, d_v, flags, eps, S0, z0, O, S_out,
                        z_out, chunk, ws, need > 0 ? (size_t)LA_NOALLOC_SCRATCH_BYTES : 0,
                        dev_status, stream);
}

}  // extern "C"
