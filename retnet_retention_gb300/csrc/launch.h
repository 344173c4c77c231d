// Internal launch interface between the C ABI (abi.cu) and the kernels.
// Nothing here is exported from liblinattn.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace la {

// Arguments of one chunkwise forward, already validated by the ABI layer.
struct ChunkArgs {
    const void* Q;
    const void* K;
    const void* V;
    void* O;
    const float* S0;  // may be null
    const float* z0;  // may be null
    float* S_out;     // may be null
    float* z_out;     // may be null
    int B, H, T, dk, dv;
    int chunk;        // requested chunk length (0 = auto)
    bool bf16;
    bool phi;
    bool normalize;
    bool floor_norm;  // divide by max(|phi(q)^T z|, 1) (normalize is set too)
    bool noncausal;
    // second-order Taylor feature map: q, k of width dk = 16, states of
    // 1 + dk + dk^2 rows in the page's feature order
    bool taylor;
    float eps;
    // per-token decay: device fp32 [B][H][T] natural logs, in place of the per-head
    // gammas (null: the gammas)
    const float* log_a;
    void* workspace;
    size_t workspace_bytes;
    int* dev_status;
    // reversed time: o_t = q_t S'_t with S'_t = gamma S'_{t+1} + k_t^T v_t, the
    // initial state entering after the last token and S_out the state after the
    // first (plain retention with the factored decay only; tc_reverse_supported)
    bool reverse = false;
    // Segment contributions of a segmented launch ([BH][segments][dk][dv] fp32):
    // where the state walk writes them (null: the workspace), or, with agg_ready,
    // already there (from a launch with the same segment plan), so that the state
    // walk is skipped (no normaliser, no z, no per-token decay).
    float* agg = nullptr;
    bool agg_ready = false;
    // Rows of Q and K stored qk_cols wide, qk_pitch elements apart (0: d_k), of V
    // v_pitch apart (0: d_v) (pipelined kernel): columns from qk_cols up to d_k are
    // read as zeros.
    int qk_cols = 0, qk_pitch = 0, v_pitch = 0;
};

struct StepArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* S;
    float* z;  // null unless normalising
    int B, H, dk, dv;
    bool bf16;
    bool phi;
    bool normalize;
    bool floor_norm;  // divide by max(|phi(q)^T z|, 1) (normalize is set too)
    float eps;
    const float* log_a;  // per-token decay: device fp32 [B][H] natural logs, or null
    bool taylor;         // Taylor feature map: dk = 16 wide q, k; states of 1 + dk + dk^2 rows
};

// Arguments of one backward pass (gradients), validated by the ABI layer.
struct BwdArgs {
    const void* Q;
    const void* K;
    const void* V;
    const void* dO;
    const float* S0;    // may be null
    const float* z0;    // may be null
    const float* dS_T;  // may be null (zero)
    const float* dz_T;  // may be null (zero)
    void* dQ;
    void* dK;
    void* dV;
    float* dS0;         // may be null
    float* dz0;         // may be null
    int B, H, T, dk, dv;
    bool bf16;
    bool phi;
    bool normalize;
    bool floor_norm;
    float eps;
    const float* log_a;  // per-token decay, or null
    bool taylor;         // Taylor feature map: dk = 16 wide q, k; states of 1 + dk + dk^2 rows
    void* workspace;     // the forward sweep's per-token den, du (normalising)
    size_t workspace_bytes;
    // the CUDA-core kernel's forward sweep alone: dq and (normalising) the per-token
    // dd, du at bwd_stats_offset in the workspace; dk, dv and the state gradients
    // are left to the caller
    bool dq_only = false;
};

// The test and diagnostic switches of la_debug_set (abi.cu).
int opt_path();           // 0 automatic, 1 CUDA cores, 2 tensor cores
bool opt_tc_lockstep();   // the lockstep kernel instead of the pipelined one
bool opt_force_timeout(); // the kernels' forced 1 ms wait and timeout status

// Normaliser mode passed to the kernels: 0 none, 1 divide by phi(q)^T z + eps,
// 2 divide by max(|phi(q)^T z|, 1).
inline int norm_mode(bool normalize, bool floor_norm) { return normalize ? (floor_norm ? 2 : 1) : 0; }

// state.cu
cudaError_t launch_state_zero(float* S, float* z, size_t n_S, size_t n_z, cudaStream_t s);
cudaError_t launch_state_copy(float* dst, const float* src, size_t n, cudaStream_t s);

// decode.cu
cudaError_t launch_decode_step(const StepArgs& a, const KernelGammas& g, cudaStream_t s);

// chunk_simt.cu: the fp32 SIMT chunkwise kernel (any supported shape)
cudaError_t launch_chunk_simt(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s);
int simt_chunk_len(int requested, int dk);

// chunk_bwd_simt.cu: the backward pass on the CUDA cores (d_k, d_v <= 128); long
// sequences are cut into segments (workspace: per-token denominators when
// normalising, the segments' states)
cudaError_t launch_chunk_bwd_simt(const BwdArgs& a, const KernelGammas& g, cudaStream_t s);
size_t bwd_workspace_bytes(const BwdArgs& a);
// Byte offset in the CUDA-core kernel's workspace of its per-token [B][H][T][2] dd, du.
size_t bwd_stats_offset(const BwdArgs& a);

// chunk_bwd_tc.cu: the backward pass as three forward passes on the tensor cores
// (bf16, no feature map, no normaliser, per-head decay, d_k, d_v in {64, 128})
bool bwd_tc_supported(const BwdArgs& a);
size_t bwd_tc_workspace_bytes(const BwdArgs& a);
cudaError_t launch_chunk_bwd_tc(const BwdArgs& a, const KernelGammas& g, cudaStream_t s);

// chunk_tc.cu: the tcgen05 chunkwise kernels (bf16, d_k in {64,128}, d_v in {64,128,256})
bool tc_supported(const ChunkArgs& a);
bool tc_reverse_supported(const ChunkArgs& a, const KernelGammas& g);
// The segment plan of a tensor-core call: segments per sequence (1: none) and
// chunks per segment.
void tc_segments(const ChunkArgs& a, int* n_seg, int* seg_chunks);
size_t tc_workspace_bytes(const ChunkArgs& a);
// Kernel launches of one tensor-core chunkwise call (1 to 4).
int tc_launch_count(const ChunkArgs& a);
cudaError_t launch_chunk_tc(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s,
                            int* launches);

// chunk_taylor.cu: causal attention with the Taylor feature map (bf16, d_k = 16,
// d_v a multiple of 64), features built on chip
bool taylor_supported(const ChunkArgs& a);
int taylor_feature_dim(int d);
cudaError_t launch_chunk_taylor(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s);

}  // namespace la
