// The exported C ABI of liblinattn.so (declared in include/linattn.h):
// argument checks on the host, then asynchronous launches on the caller's
// stream.  Nothing is launched or written when a check fails.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "launch.h"

using namespace la;

namespace {
// la_debug_set's switches (indexed by LA_OPT_*)
std::atomic<int> g_opt[4] = {};
}  // namespace

namespace la {
int opt_path() { return g_opt[LA_OPT_PATH].load(std::memory_order_relaxed); }
bool opt_tc_lockstep() { return g_opt[LA_OPT_TC_LOCKSTEP].load(std::memory_order_relaxed) != 0; }
bool opt_force_timeout() { return g_opt[LA_OPT_FORCE_TIMEOUT].load(std::memory_order_relaxed) != 0; }
}  // namespace la

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dim(int d) { return d >= 16 && d <= 256 && d % 16 == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

// Fills the per-head decay block; returns false if any gamma is outside (0, 1].
bool fill_gammas(const float* gamma, int H, KernelGammas* g, bool* all_one) {
    std::memset(g, 0, sizeof(*g));
    *all_one = true;
    for (int h = 0; h < H; ++h) {
        float x = gamma[h];
        if (!(x > 0.f && x <= 1.f)) return false;  // also rejects NaN
        g->gamma[h] = x;
        g->log2g[h] = (float)std::log2((double)x);
        if (x != 1.f) *all_one = false;
    }
    return true;
}

const float kOneGamma = 1.f;  // stands in for an absent gamma array when B * H == 0

la_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

size_t elem_size(la_dtype dt) { return dt == LA_DTYPE_BF16 ? 2 : 4; }

constexpr unsigned kCallFlags = LA_PHI_ELU1 | LA_NORMALIZE | LA_NONCAUSAL | LA_NORM_FLOOR;

// The arguments la_chunk_fwd's path choice depends on (pointers are irrelevant;
// a per-token decay is marked by a non-null log_a).
ChunkArgs plan_args(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags,
                    int chunk) {
    static const float kMarker = 0.f;
    ChunkArgs a;
    std::memset(&a, 0, sizeof(a));
    a.B = B; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v; a.chunk = chunk;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.phi = (flags & LA_PHI_ELU1) != 0;
    a.normalize = (flags & (LA_NORMALIZE | LA_NORM_FLOOR)) != 0;
    a.floor_norm = (flags & LA_NORM_FLOOR) != 0;
    a.noncausal = (flags & LA_NONCAUSAL) != 0;
    a.taylor = (flags & LA_PHI_TAYLOR) != 0;
    a.log_a = (flags & LA_GATED) ? &kMarker : nullptr;
    return a;
}

bool plan_ok(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags) {
    return B > 0 && H > 0 && T > 0 && valid_dim(d_k) && valid_dim(d_v) && H <= kMaxHeads &&
           (dtype == LA_DTYPE_F32 || dtype == LA_DTYPE_BF16) &&
           !(flags & ~(kCallFlags | LA_GATED | LA_PHI_TAYLOR));
}

bool simt_pinned() { return opt_path() == 1; }

// The backward pass's path: the tensor cores (three forward passes) where they
// apply, unless LA_OPT_PATH pins the CUDA-core kernel.
BwdArgs bwd_plan_args(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags,
                      bool gated) {
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    static const float kMarker = 0.f;
    a.B = B; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.phi = (flags & LA_PHI_ELU1) != 0;
    a.floor_norm = (flags & LA_NORM_FLOOR) != 0;
    a.normalize = (flags & LA_NORMALIZE) != 0 || a.floor_norm;
    a.log_a = gated ? &kMarker : nullptr;
    a.taylor = (flags & LA_PHI_TAYLOR) != 0;
    return a;
}

size_t bwd_bytes_for(const BwdArgs& a) {
    if (!simt_pinned() && bwd_tc_supported(a)) return bwd_tc_workspace_bytes(a);
    return bwd_workspace_bytes(a);
}

}  // namespace

extern "C" {

const char* la_status_string(int status) {
    switch (status) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported combination";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

int la_abi_version(void) { return LA_ABI_VERSION; }

int la_debug_set(int option, int value) {
    const int hi = option == LA_OPT_PATH ? 2 : 1;
    if (option < LA_OPT_PATH || option > LA_OPT_FORCE_TIMEOUT || value < 0 || value > hi) return -1;
    return g_opt[option].exchange(value);
}

size_t la_workspace_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags,
                         int chunk) {
    if (!plan_ok(B, H, T, d_k, d_v, dtype, flags)) return 0;
    ChunkArgs a = plan_args(B, H, T, d_k, d_v, dtype, flags, chunk);
    if (simt_pinned() || !tc_supported(a)) return 0;
    return tc_workspace_bytes(a);
}

int la_chunk_fwd_launches(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags,
                          int chunk) {
    if (!plan_ok(B, H, T, d_k, d_v, dtype, flags)) return 0;
    ChunkArgs a = plan_args(B, H, T, d_k, d_v, dtype, flags, chunk);
    if (simt_pinned() || !tc_supported(a)) return 1;
    return tc_launch_count(a);
}

la_status la_state_init(float* S, float* z, int B, int H, int d_k, int d_v, la_stream_t stream) {
    if (B < 0 || H < 0 || !valid_dim(d_k) || !valid_dim(d_v)) return LA_ERR_INVALID_ARG;
    if ((size_t)B * H == 0) return LA_OK;
    if (!S || !aligned16(S) || (z && !aligned16(z))) return LA_ERR_INVALID_ARG;
    const size_t nbh = (size_t)B * H;
    return cuda_status(launch_state_zero(S, z, nbh * d_k * d_v, z ? nbh * d_k : 0,
                                         (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// la_chunk_fwd and la_chunk_fwd_gated: exactly one of gamma (host [H]) and log_a
// (device [B][H][T]) is given.  check_only: return after the checks, launching
// nothing.
la_status chunk_fwd(const void* Q, const void* K, const void* V, la_dtype dtype,
                    const float* gamma, const float* log_a, int B, int H, int T, int d_k,
                    int d_v, unsigned flags, float eps, const float* S0, const float* z0,
                    void* O, float* S_out, float* z_out, int chunk, void* workspace,
                    size_t workspace_bytes, int* dev_status, la_stream_t stream,
                    bool check_only = false) {
    const bool gated = gamma == nullptr;
    if (B < 0 || H < 0 || T < 0 || !valid_dim(d_k) || !valid_dim(d_v)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16) return LA_ERR_INVALID_ARG;
    if (flags & ~(kCallFlags | LA_PHI_TAYLOR | (gated ? LA_GATED : 0u))) return LA_ERR_INVALID_ARG;
    const bool taylor = (flags & LA_PHI_TAYLOR) != 0;
    if (taylor && (gated || dtype != LA_DTYPE_BF16 || d_k != 16 || d_v % 64 != 0 ||
                   (flags & (LA_PHI_ELU1 | LA_NONCAUSAL)) || !(chunk == 0 || chunk == 128)))
        return LA_ERR_UNSUPPORTED;
    if (!(chunk == 0 || chunk == 16 || chunk == 32 || chunk == 64 || chunk == 128))
        return LA_ERR_INVALID_ARG;
    if (H > kMaxHeads) return LA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
    const size_t nbh = (size_t)B * H;
    if (nbh == 0) return LA_OK;
    KernelGammas g;
    bool all_one = true;
    if (gated) {
        std::memset(&g, 0, sizeof(g));
        all_one = false;
    } else if (!fill_gammas(gamma, H, &g, &all_one)) {
        return LA_ERR_INVALID_ARG;
    }
    const bool noncausal = (flags & LA_NONCAUSAL) != 0;
    const bool floor_norm = (flags & LA_NORM_FLOOR) != 0;
    const bool normalize = (flags & LA_NORMALIZE) != 0 || floor_norm;
    if (noncausal && (gated || !all_one || S0 || z0)) return LA_ERR_UNSUPPORTED;

    const size_t es = elem_size(dtype);
    const size_t n_qk = nbh * (size_t)T * d_k * es, n_v = nbh * (size_t)T * d_v * es;
    if (T > 0) {
        if (!Q || !K || !V || !O) return LA_ERR_INVALID_ARG;
        if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
            return LA_ERR_INVALID_ARG;
        if (overlaps(O, n_v, Q, n_qk) || overlaps(O, n_v, K, n_qk) || overlaps(O, n_v, V, n_v))
            return LA_ERR_INVALID_ARG;
        if (gated && (!log_a || !aligned16(log_a) || overlaps(O, n_v, log_a, nbh * T * 4)))
            return LA_ERR_INVALID_ARG;
    }
    for (const void* p : {(const void*)S0, (const void*)z0, (const void*)S_out,
                          (const void*)z_out, (const void*)workspace})
        if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
    if (workspace_bytes <
        la_workspace_size(B, H, T, d_k, d_v, dtype, flags | (gated ? LA_GATED : 0u), chunk))
        return LA_ERR_INVALID_ARG;

    cudaStream_t s = (cudaStream_t)stream;
    const size_t ds = taylor ? (size_t)taylor_feature_dim(d_k) : (size_t)d_k;  // state rows
    const size_t nS = nbh * ds * d_v, nz = nbh * ds;
    if (T == 0) {  // empty sequence: the final state is the initial one
        if (check_only) return LA_OK;
        cudaError_t e = cudaSuccess;
        if (S_out) e = S0 ? launch_state_copy(S_out, S0, nS, s) : launch_state_zero(S_out, nullptr, nS, 0, s);
        if (e == cudaSuccess && z_out)
            e = z0 ? launch_state_copy(z_out, z0, nz, s) : launch_state_zero(z_out, nullptr, nz, 0, s);
        return cuda_status(e);
    }

    ChunkArgs a;
    a.Q = Q; a.K = K; a.V = V; a.O = O;
    a.S0 = S0; a.z0 = z0; a.S_out = S_out; a.z_out = z_out;
    a.B = B; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v;
    a.chunk = chunk;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.phi = (flags & LA_PHI_ELU1) != 0;
    a.normalize = normalize;
    a.floor_norm = floor_norm;
    a.noncausal = noncausal;
    a.taylor = taylor;
    a.eps = eps;
    a.log_a = gated ? log_a : nullptr;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.dev_status = dev_status;
    // LA_OPT_PATH pins the path (tests compare both); default: tensor cores
    // whenever the shape allows, the fp32 CUDA-core kernel otherwise.
    const bool want_simt = opt_path() == 1;
    const bool want_tc = opt_path() == 2;
    if (taylor) {  // its own tensor-core kernel; no CUDA-core version
        if (want_simt || !taylor_supported(a)) return LA_ERR_UNSUPPORTED;
        return check_only ? LA_OK : cuda_status(launch_chunk_taylor(a, g, s));
    }
    if (!want_simt && tc_supported(a)) {
        int launches = 0;
        return check_only ? LA_OK : cuda_status(launch_chunk_tc(a, g, s, &launches));
    }
    if (want_tc) return LA_ERR_UNSUPPORTED;
    return check_only ? LA_OK : cuda_status(launch_chunk_simt(a, g, s));
}

la_status recurrent_step(const void* q, const void* k, const void* v, la_dtype dtype,
                         const float* gamma, const float* log_a, int B, int H, int d_k, int d_v,
                         unsigned flags, float eps, float* S, float* z, void* o,
                         la_stream_t stream) {
    const bool gated = gamma == nullptr;
    if (B < 0 || H < 0 || !valid_dim(d_k) || !valid_dim(d_v)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16) return LA_ERR_INVALID_ARG;
    if (flags & ~(kCallFlags | LA_PHI_TAYLOR | (gated ? LA_GATED : 0u))) return LA_ERR_INVALID_ARG;
    if (flags & LA_NONCAUSAL) return LA_ERR_UNSUPPORTED;
    const bool taylor = (flags & LA_PHI_TAYLOR) != 0;
    if (taylor && (d_k != 16 || (flags & LA_PHI_ELU1))) return LA_ERR_UNSUPPORTED;
    const size_t ds = taylor ? (size_t)taylor_feature_dim(d_k) : (size_t)d_k;  // state rows
    if (H > kMaxHeads) return LA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
    const size_t nbh = (size_t)B * H;
    if (nbh == 0) return LA_OK;
    KernelGammas g;
    bool all_one = true;
    if (gated) {
        std::memset(&g, 0, sizeof(g));
    } else if (!fill_gammas(gamma, H, &g, &all_one)) {
        return LA_ERR_INVALID_ARG;
    }
    const bool floor_norm = (flags & LA_NORM_FLOOR) != 0;
    const bool normalize = (flags & LA_NORMALIZE) != 0 || floor_norm;
    if (!q || !k || !v || !o || !S || (normalize && !z) || (gated && !log_a))
        return LA_ERR_INVALID_ARG;
    for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o,
                          (const void*)S, (const void*)z, (const void*)log_a})
        if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    const size_t n_o = nbh * d_v * es;
    if (overlaps(o, n_o, q, nbh * d_k * es) || overlaps(o, n_o, k, nbh * d_k * es) ||
        overlaps(o, n_o, v, n_o) || overlaps(o, n_o, S, nbh * ds * d_v * 4))
        return LA_ERR_INVALID_ARG;

    StepArgs a;
    a.taylor = taylor;
    a.q = q; a.k = k; a.v = v; a.o = o; a.S = S; a.z = normalize ? z : nullptr;
    a.B = B; a.H = H; a.dk = d_k; a.dv = d_v;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.phi = (flags & LA_PHI_ELU1) != 0;
    a.normalize = normalize;
    a.floor_norm = floor_norm;
    a.eps = eps;
    a.log_a = gated ? log_a : nullptr;
    return cuda_status(launch_decode_step(a, g, (cudaStream_t)stream));
}

la_status chunk_bwd(const void* Q, const void* K, const void* V, const void* dO, la_dtype dtype,
                    const float* gamma, const float* log_a, int B, int H, int T, int d_k,
                    int d_v, unsigned flags, float eps, const float* S0, const float* z0,
                    const float* dS_T, const float* dz_T, void* dQ, void* dK, void* dV,
                    float* dS0, float* dz0, void* workspace, size_t workspace_bytes,
                    la_stream_t stream) {
    const bool gated = gamma == nullptr;
    const bool taylor = (flags & LA_PHI_TAYLOR) != 0;
    if (B < 0 || H < 0 || T < 0 || !valid_dim(d_k) || !valid_dim(d_v)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16) return LA_ERR_INVALID_ARG;
    if (flags & ~(kCallFlags | LA_PHI_TAYLOR | (gated ? LA_GATED : 0u))) return LA_ERR_INVALID_ARG;
    // the Taylor map: 16-wide q and k, per-head decay, not with elu + 1
    if (taylor && (gated || d_k != 16 || (flags & LA_PHI_ELU1))) return LA_ERR_UNSUPPORTED;
    if (H > kMaxHeads) return LA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
    const size_t nbh = (size_t)B * H;
    if (nbh == 0) return LA_OK;
    KernelGammas g;
    bool all_one = true;
    if (gated) {
        std::memset(&g, 0, sizeof(g));
    } else if (!fill_gammas(gamma, H, &g, &all_one)) {
        return LA_ERR_INVALID_ARG;
    }
    if (flags & LA_NONCAUSAL) return LA_ERR_UNSUPPORTED;
    if (d_k > 128 || d_v > 128) return LA_ERR_UNSUPPORTED;
    const bool floor_norm = (flags & LA_NORM_FLOOR) != 0;
    const bool normalize = (flags & LA_NORMALIZE) != 0 || floor_norm;
    const size_t es = elem_size(dtype);
    const size_t n_qk = nbh * (size_t)T * d_k * es, n_v = nbh * (size_t)T * d_v * es;
    if (T > 0) {
        if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return LA_ERR_INVALID_ARG;
        for (const void* p : {Q, K, V, dO, (const void*)dQ, (const void*)dK, (const void*)dV})
            if (!aligned16(p)) return LA_ERR_INVALID_ARG;
        if (gated && (!log_a || !aligned16(log_a))) return LA_ERR_INVALID_ARG;
        const void* ins[5] = {Q, K, V, dO, log_a};
        const size_t nin[5] = {n_qk, n_qk, n_v, n_v, gated ? nbh * T * 4 : 0};
        const void* outs[3] = {dQ, dK, dV};
        const size_t nout[3] = {n_qk, n_qk, n_v};
        for (int o = 0; o < 3; ++o) {
            for (int i = 0; i < 5; ++i)
                if (overlaps(outs[o], nout[o], ins[i], nin[i])) return LA_ERR_INVALID_ARG;
            for (int o2 = o + 1; o2 < 3; ++o2)
                if (overlaps(outs[o], nout[o], outs[o2], nout[o2])) return LA_ERR_INVALID_ARG;
        }
    }
    for (const void* p : {(const void*)S0, (const void*)z0, (const void*)dS_T, (const void*)dz_T,
                          (const void*)dS0, (const void*)dz0, (const void*)workspace})
        if (p && !aligned16(p)) return LA_ERR_INVALID_ARG;
    const size_t need = T > 0 ? bwd_bytes_for(bwd_plan_args(B, H, T, d_k, d_v, dtype, flags, gated)) : 0;
    if (workspace_bytes < need || (need > 0 && !workspace)) return LA_ERR_INVALID_ARG;

    BwdArgs a;
    a.Q = Q; a.K = K; a.V = V; a.dO = dO;
    a.S0 = S0; a.z0 = z0; a.dS_T = dS_T; a.dz_T = dz_T;
    a.dQ = dQ; a.dK = dK; a.dV = dV; a.dS0 = dS0; a.dz0 = dz0;
    a.B = B; a.H = H; a.T = T; a.dk = d_k; a.dv = d_v;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.phi = (flags & LA_PHI_ELU1) != 0;
    a.normalize = normalize;
    a.floor_norm = floor_norm;
    a.eps = eps;
    a.log_a = gated ? log_a : nullptr;
    a.taylor = taylor;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    if (T > 0 && !simt_pinned() && bwd_tc_supported(a))
        return cuda_status(launch_chunk_bwd_tc(a, g, (cudaStream_t)stream));
    return cuda_status(launch_chunk_bwd_simt(a, g, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

size_t la_bwd_workspace_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype,
                             unsigned flags) {
    if (!plan_ok(B, H, T, d_k, d_v, dtype, flags) || d_k > 128 || d_v > 128) return 0;
    if ((flags & LA_PHI_TAYLOR) && (d_k != 16 || (flags & (LA_PHI_ELU1 | LA_GATED)))) return 0;
    return bwd_bytes_for(bwd_plan_args(B, H, T, d_k, d_v, dtype, flags, (flags & LA_GATED) != 0));
}

la_status la_chunk_bwd(const void* Q, const void* K, const void* V, const void* dO,
                       la_dtype dtype, const float* gamma, int B, int H, int T, int d_k, int d_v,
                       unsigned flags, float eps, const float* S0, const float* z0,
                       const float* dS_T, const float* dz_T, void* dQ, void* dK, void* dV,
                       float* dS0, float* dz0, void* workspace, size_t workspace_bytes,
                       int* dev_status, la_stream_t stream) {
    (void)dev_status;  // the backward kernels have no device-side waits
    if (!gamma && (size_t)B * H > 0 && B > 0 && H > 0) return LA_ERR_INVALID_ARG;
    if (!gamma) gamma = &kOneGamma;
    return chunk_bwd(Q, K, V, dO, dtype, gamma, nullptr, B, H, T, d_k, d_v, flags, eps, S0, z0,
                     dS_T, dz_T, dQ, dK, dV, dS0, dz0, workspace, workspace_bytes, stream);
}

la_status la_chunk_bwd_gated(const void* Q, const void* K, const void* V, const void* dO,
                             la_dtype dtype, const float* log_a, int B, int H, int T, int d_k,
                             int d_v, unsigned flags, float eps, const float* S0, const float* z0,
                             const float* dS_T, const float* dz_T, void* dQ, void* dK, void* dV,
                             float* dS0, float* dz0, void* workspace, size_t workspace_bytes,
                             int* dev_status, la_stream_t stream) {
    (void)dev_status;
    return chunk_bwd(Q, K, V, dO, dtype, nullptr, log_a, B, H, T, d_k, d_v, flags, eps, S0, z0,
                     dS_T, dz_T, dQ, dK, dV, dS0, dz0, workspace, workspace_bytes, stream);
}

la_status la_chunk_fwd(const void* Q, const void* K, const void* V, la_dtype dtype,
                       const float* gamma, int B, int H, int T, int d_k, int d_v,
                       unsigned flags, float eps, const float* S0, const float* z0, void* O,
                       float* S_out, float* z_out, int chunk, void* workspace,
                       size_t workspace_bytes, int* dev_status, la_stream_t stream) {
    if (!gamma && (size_t)B * H > 0 && B > 0 && H > 0) return LA_ERR_INVALID_ARG;
    if (!gamma) gamma = &kOneGamma;  // B or H == 0 (or negative: rejected below)
    return chunk_fwd(Q, K, V, dtype, gamma, nullptr, B, H, T, d_k, d_v, flags, eps, S0, z0, O,
                     S_out, z_out, chunk, workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"

namespace {

// The device arena of la_chunk_fwd_host: two slots (double buffering), each with
// one piece's Q, K, V, O, S0, z0, S_out, z_out and chunk workspace; byte offsets
// within a slot, every region 256-byte aligned.  A piece has at most bmax
// sequences of the batch (pieces of floor or ceil(B / pieces) rows).
struct HostPlan {
    int bmax;
    size_t o_q, o_k, o_v, o_o, o_s0, o_z0, o_so, o_zo, o_ws, ws, slot, bytes;
};

bool host_plan(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags, int chunk,
               int pieces, HostPlan* hp) {
    std::memset(hp, 0, sizeof(*hp));
    if (B < 0 || H < 0 || T < 0 || !valid_dim(d_k) || !valid_dim(d_v)) return false;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16) return false;
    if (B > 0 && (pieces < 1 || pieces > B)) return false;
    if (B == 0) return true;
    const int bmax = (B + pieces - 1) / pieces, bmin = B / pieces;
    const size_t es = elem_size(dtype);
    const size_t ds = (flags & LA_PHI_TAYLOR) ? (size_t)taylor_feature_dim(d_k) : (size_t)d_k;
    const size_t nbh = (size_t)bmax * H;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    hp->bmax = bmax;
    hp->o_q = take(nbh * T * d_k * es);
    hp->o_k = take(nbh * T * d_k * es);
    hp->o_v = take(nbh * T * d_v * es);
    hp->o_o = take(nbh * T * d_v * es);
    hp->o_s0 = take(nbh * ds * d_v * 4);
    hp->o_z0 = take(nbh * ds * 4);
    hp->o_so = take(nbh * ds * d_v * 4);
    hp->o_zo = take(nbh * ds * 4);
    // the smaller pieces can have a plan of their own (more segments per sequence)
    hp->ws = std::max(la_workspace_size(bmax, H, T, d_k, d_v, dtype, flags, chunk),
                      bmin > 0 ? la_workspace_size(bmin, H, T, d_k, d_v, dtype, flags, chunk) : 0);
    hp->o_ws = take(hp->ws);
    hp->slot = off;
    hp->bytes = 2 * off;
    return true;
}

}  // namespace

extern "C" {

size_t la_host_arena_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype, unsigned flags,
                          int chunk, int pieces) {
    HostPlan hp;
    return host_plan(B, H, T, d_k, d_v, dtype, flags, chunk, pieces, &hp) ? hp.bytes : 0;
}

la_status la_chunk_fwd_host(const void* Q, const void* K, const void* V, la_dtype dtype,
                            const float* gamma, int B, int H, int T, int d_k, int d_v,
                            unsigned flags, float eps, const float* S0, const float* z0, void* O,
                            float* S_out, float* z_out, int chunk, int pieces, void* arena,
                            size_t arena_bytes, int* dev_status, la_stream_t stream) {
    HostPlan hp;
    if (!host_plan(B, H, T, d_k, d_v, dtype, flags, chunk, pieces, &hp)) return LA_ERR_INVALID_ARG;
    if ((size_t)B * H == 0 || B <= 0 || H <= 0) return LA_OK;
    if (!gamma) return LA_ERR_INVALID_ARG;
    if (T > 0 && (!Q || !K || !V || !O)) return LA_ERR_INVALID_ARG;
    if (!arena || !aligned16(arena) || arena_bytes < hp.bytes) return LA_ERR_INVALID_ARG;
    char* slot[2] = {static_cast<char*>(arena), static_cast<char*>(arena) + hp.slot};
    auto dev = [&](int sl, size_t o) { return static_cast<void*>(slot[sl] + o); };
    // every check of the per-piece calls, before anything is enqueued
    la_status st = chunk_fwd(dev(0, hp.o_q), dev(0, hp.o_k), dev(0, hp.o_v), dtype, gamma, nullptr,
                             hp.bmax, H, T, d_k, d_v, flags, eps,
                             S0 ? (const float*)dev(0, hp.o_s0) : nullptr,
                             z0 ? (const float*)dev(0, hp.o_z0) : nullptr, dev(0, hp.o_o),
                             S_out ? (float*)dev(0, hp.o_so) : nullptr,
                             z_out ? (float*)dev(0, hp.o_zo) : nullptr, chunk, dev(0, hp.o_ws),
                             hp.ws, dev_status, stream, /*check_only=*/true);
    if (st != LA_OK) return st;

    const size_t es = elem_size(dtype);
    const size_t ds = (flags & LA_PHI_TAYLOR) ? (size_t)taylor_feature_dim(d_k) : (size_t)d_k;
    const size_t row_qk = (size_t)H * T * d_k * es, row_v = (size_t)H * T * d_v * es;
    const size_t row_s = (size_t)H * ds * d_v * 4, row_z = (size_t)H * ds * 4;
    cudaStream_t main = (cudaStream_t)stream;
    cudaStream_t ss[2] = {nullptr, nullptr};
    cudaEvent_t start = nullptr, done[2] = {nullptr, nullptr};
    cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    for (int j = 0; j < 2 && e == cudaSuccess; ++j) {
        e = cudaStreamCreateWithFlags(&ss[j], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[j], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventRecord(start, main);
    for (int j = 0; j < 2 && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(ss[j], start, 0);
    // piece i: copy in, forward, copy out, in order on stream i mod 2 (slot i mod 2),
    // so piece i + 1's copies overlap piece i's compute and slot reuse is ordered
    for (int i = 0; i < pieces && e == cudaSuccess && st == LA_OK; ++i) {
        const int b0 = (int)(((long long)i * B) / pieces), b1 = (int)(((long long)(i + 1) * B) / pieces);
        const int b = b1 - b0, sl = i & 1;
        cudaStream_t s = ss[sl];
        auto h2d = [&](size_t o, const void* src, size_t row) {
            if (e == cudaSuccess && src)
                e = cudaMemcpyAsync(dev(sl, o), static_cast<const char*>(src) + (size_t)b0 * row,
                                    (size_t)b * row, cudaMemcpyHostToDevice, s);
        };
        auto d2h = [&](void* dst, size_t o, size_t row) {
            if (e == cudaSuccess && dst)
                e = cudaMemcpyAsync(static_cast<char*>(dst) + (size_t)b0 * row, dev(sl, o),
                                    (size_t)b * row, cudaMemcpyDeviceToHost, s);
        };
        h2d(hp.o_q, Q, row_qk);
        h2d(hp.o_k, K, row_qk);
        h2d(hp.o_v, V, row_v);
        h2d(hp.o_s0, S0, row_s);
        h2d(hp.o_z0, z0, row_z);
        if (e != cudaSuccess) break;
        st = chunk_fwd(dev(sl, hp.o_q), dev(sl, hp.o_k), dev(sl, hp.o_v), dtype, gamma, nullptr, b, H,
                       T, d_k, d_v, flags, eps, S0 ? (const float*)dev(sl, hp.o_s0) : nullptr,
                       z0 ? (const float*)dev(sl, hp.o_z0) : nullptr, dev(sl, hp.o_o),
                       S_out ? (float*)dev(sl, hp.o_so) : nullptr,
                       z_out ? (float*)dev(sl, hp.o_zo) : nullptr, chunk, dev(sl, hp.o_ws), hp.ws,
                       dev_status, (la_stream_t)s);
        d2h(O, hp.o_o, row_v);
        d2h(S_out, hp.o_so, row_s);
        d2h(z_out, hp.o_zo, row_z);
    }
    // the caller's stream waits for both pipelines; the streams and events are
    // released once their work completes
    for (int j = 0; j < 2; ++j) {
        if (ss[j] && done[j] && cudaEventRecord(done[j], ss[j]) == cudaSuccess)
            cudaStreamWaitEvent(main, done[j], 0);
        if (done[j]) cudaEventDestroy(done[j]);
        if (ss[j]) cudaStreamDestroy(ss[j]);
    }
    if (start) cudaEventDestroy(start);
    if (st != LA_OK) return st;
    return cuda_status(e);
}

la_status la_chunk_fwd_gated(const void* Q, const void* K, const void* V, la_dtype dtype,
                             const float* log_a, int B, int H, int T, int d_k, int d_v,
                             unsigned flags, float eps, const float* S0, const float* z0,
                             void* O, float* S_out, float* z_out, int chunk, void* workspace,
                             size_t workspace_bytes, int* dev_status, la_stream_t stream) {
    return chunk_fwd(Q, K, V, dtype, nullptr, log_a, B, H, T, d_k, d_v, flags, eps, S0, z0, O,
                     S_out, z_out, chunk, workspace, workspace_bytes, dev_status, stream);
}

la_status la_recurrent_step(const void* q, const void* k, const void* v, la_dtype dtype,
                            const float* gamma, int B, int H, int d_k, int d_v, unsigned flags,
                            float eps, float* S, float* z, void* o, int* dev_status,
                            la_stream_t stream) {
    (void)dev_status;  // the decode step has no device-side waits
    if (!gamma && (size_t)B * H > 0 && B > 0 && H > 0) return LA_ERR_INVALID_ARG;
    if (!gamma) gamma = &kOneGamma;
    return recurrent_step(q, k, v, dtype, gamma, nullptr, B, H, d_k, d_v, flags, eps, S, z, o,
                          stream);
}

la_status la_recurrent_step_gated(const void* q, const void* k, const void* v, la_dtype dtype,
                                  const float* log_a, int B, int H, int d_k, int d_v,
                                  unsigned flags, float eps, float* S, float* z, void* o,
                                  int* dev_status, la_stream_t stream) {
    (void)dev_status;
    return recurrent_step(q, k, v, dtype, nullptr, log_a, B, H, d_k, d_v, flags, eps, S, z, o,
                          stream);
}

}  // extern "C"
