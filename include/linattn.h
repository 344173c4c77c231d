/*
 * linattn.h - C ABI of the GB300 (sm_103a) causal decayed linear attention
 * library, liblinattn.so.
 *
 * The operator (one head, one sequence):
 *
 *   S_t = gamma * S_{t-1} + phi(k_t) v_t^T        S: d_k x d_v, fp32
 *   z_t = gamma * z_{t-1} + phi(k_t)              z: d_k,       fp32
 *   o_t = phi(q_t)^T S_t  [ / (phi(q_t)^T z_t + eps)  when normalising ]
 *
 * which equals the masked parallel form O = (Q K^T . D) V, D_nm = gamma^(n-m)
 * for n >= m and 0 otherwise.
 *   - "RetNet" (bembew): "Parallel Representation" (O = (QK^T . D)V and D),
 *     "Recurrent Representation" (S_n = gamma S_{n-1} + K_n^T V_n,
 *     O_n = Q_n S_n), "Chunked Recurrent Representation" (chunks computed in
 *     parallel, the state carried between them), "Multi-Scale Retention"
 *     (one gamma per head).
 *   - "Linear attention" (zerotofrontier 21.2): box "Causal linear attention,
 *     recurrent form" (phi, the normaliser z, eps in the denominator, rows of
 *     S index features and columns value dimensions) and box "Linear
 *     attention" (the non-causal form).
 *   - "Efficient and Sparse Transformers" (temporalbook 12.5), subsection 6:
 *     linear attention is the gamma = 1 case; phi(x) = elu(x) + 1.
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major, caller-owned DEVICE memory (allocated by
 *     the caller, e.g. PyTorch); the library allocates nothing, keeps no
 *     state between calls and never synchronises the stream.
 *   - Layouts: Q, K [B][H][T][d_k]; V, O [B][H][T][d_v]; S [B][H][d_k][d_v]
 *     (rows = features, columns = value dims); z [B][H][d_k].
 *   - Q/K/V/O hold `dtype` elements (fp32 or bf16); states are always fp32.
 *   - Every device pointer must be 16-byte aligned; d_k and d_v must be
 *     multiples of 16 in [16, 256].
 *   - `gamma` is a HOST array of H fp32 decays, each in (0, 1]; it is read
 *     during the call (its values travel in the kernel parameters), so the
 *     array may be reused as soon as the call returns.
 *   - Calls run on the CURRENT device (cudaSetDevice): it must own `stream`
 *     and every buffer passed; the segment plans and workspace sizes are the
 *     current device's too (its SM count).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  The return code covers host-side argument
 *     checks and launch errors only.  `dev_status`, if not NULL, is a device
 *     int the kernels set to a nonzero la_status when they detect a problem
 *     on the device (a bounded wait that ran out); the caller zeroes it
 *     beforehand and reads it after synchronising.
 *   - Arguments are checked before anything is enqueued: a call that returns
 *     LA_ERR_INVALID_ARG or LA_ERR_UNSUPPORTED has launched nothing and
 *     written nothing.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library (the library is built with hidden default
 * visibility; only these are exported). */
#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* bad size, pointer, alignment, gamma or workspace */
    LA_ERR_UNSUPPORTED = 2,  /* a combination the method does not define */
    LA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    LA_ERR_TIMEOUT = 4       /* device side only: a bounded wait ran out */
} la_status;

typedef enum { LA_DTYPE_F32 = 0, LA_DTYPE_BF16 = 1 } la_dtype;

/* flags */
#define LA_PHI_ELU1  1u  /* apply phi(x) = elu(x) + 1 to q and k (not v) */
#define LA_NORMALIZE 2u  /* divide by phi(q)^T z + eps */
#define LA_NONCAUSAL 4u  /* every query reads the whole sequence; gamma must be 1 */
/* Divide by max(|phi(q)^T z|, 1) instead of phi(q)^T z + eps (implies normalising;
 * eps unused): the matrix LSTM's floored normaliser, box "An LSTM whose cell is
 * linear attention" on the "Linear attention" page, which equals RetNet's
 * division of each score row by the absolute value of its sum clamped below at 1
 * (same page, "Its normalizer is unstable").  Defined for signed features too. */
#define LA_NORM_FLOOR 8u
/* Per-token decay (la_chunk_fwd_gated): only the planning queries
 * la_workspace_size and la_chunk_fwd_launches take this flag, to size a
 * la_chunk_fwd_gated call; la_chunk_fwd rejects it. */
#define LA_GATED 16u
/* Second-order Taylor feature map in place of elu + 1 ("Linear attention" page,
 * section "A Taylor feature map", box "Taylor features"):
 *   phi(x) = (1, x_1 .. x_d, vec(x x^T) / sqrt 2),  1 + d + d^2 entries, vec row-major,
 * so that phi(q)^T phi(k) = 1 + s + s^2/2 with s = q^T k (always >= 1/2, a safe
 * denominator).  d_k = 16 (Based's projected width: 273 features), not with
 * LA_PHI_ELU1, causal.  d_k is the width of Q and K; the states S0 / S_out / S are
 * [B][H][1 + d_k + d_k^2][d_v] fp32 and z0 / z_out / z [B][H][1 + d_k + d_k^2],
 * rows in the order of phi above.  la_chunk_fwd (and la_workspace_size,
 * la_chunk_fwd_launches, la_chunk_fwd_noalloc): bf16, d_v a multiple of 64, chunk
 * 0 or 128, an sm_103 device.  la_recurrent_step: bf16 or fp32, d_v <= 256.
 * la_chunk_bwd: bf16 or fp32, d_v <= 128, per-head decay.  Other calls and
 * shapes answer LA_ERR_UNSUPPORTED. */
#define LA_PHI_TAYLOR 32u

/* Human-readable text of a status code (static storage, never NULL). */
LA_API const char* la_status_string(int status);

/* ABI version of this header: LA_ABI_VERSION. */
#define LA_ABI_VERSION 1
LA_API int la_abi_version(void);

/*
 * Bytes of device workspace la_chunk_fwd needs for these arguments (0 when
 * the chosen path needs none).  Pure host arithmetic; never fails (returns
 * 0 for arguments la_chunk_fwd would reject).  `chunk` as for la_chunk_fwd.
 */
LA_API size_t la_workspace_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype,
                                unsigned flags, int chunk);

/*
 * Number of kernels la_chunk_fwd enqueues for these arguments on the current
 * device (1 for the single-pass paths; 2 or 3 when long sequences are split
 * into segments: segment states, then - for more than four segments per
 * sequence - the scan over them, then the outputs).  LA_GATED adds the decays'
 * preparation.  0 for
 * arguments la_chunk_fwd would reject or T == 0.  Pure host query.
 */
LA_API int la_chunk_fwd_launches(int B, int H, int T, int d_k, int d_v, la_dtype dtype,
                                 unsigned flags, int chunk);

/*
 * Zero-fill a state: S[B][H][d_k][d_v] and, if not NULL, z[B][H][d_k].
 * The empty state S_0 = 0, z_0 = 0 of the "Causal linear attention,
 * recurrent form" box ("Linear attention", zerotofrontier 21.2).
 * Errors: LA_ERR_INVALID_ARG for S == NULL, a negative size, or a misaligned
 * pointer; LA_ERR_CUDA if the launch fails.  B or H == 0 is a no-op.
 */
LA_API la_status la_state_init(float* S, float* z, int B, int H, int d_k, int d_v,
                               la_stream_t stream);

/*
 * Chunkwise forward over whole sequences (prefill / training forward):
 * "Chunked Recurrent Representation" ("RetNet", bembew) - the intra-chunk
 * part in the parallel form, the inter-chunk part through the carried state.
 *
 *   Q, K      [B][H][T][d_k]  dtype      inputs, read only
 *   V         [B][H][T][d_v]  dtype      input, read only
 *   gamma     host float[H]              per-head decay in (0, 1]
 *   flags     LA_PHI_ELU1 | LA_NORMALIZE | LA_NONCAUSAL | LA_NORM_FLOOR
 *   eps       added to the denominator (used only with LA_NORMALIZE and not
 *             LA_NORM_FLOOR; the pages use 1e-6)
 *   S0, z0    [B][H][d_k][d_v], [B][H][d_k] fp32 initial state, or NULL for
 *             zero.  S0 may alias S_out and z0 may alias z_out (in-place
 *             continuation).  The normaliser state z is carried whether or
 *             not LA_NORMALIZE is set, so z_out is valid either way.
 *   O         [B][H][T][d_v]  dtype      output; must not overlap Q, K, V
 *   S_out     [B][H][d_k][d_v] fp32 final state S_T, or NULL
 *   z_out     [B][H][d_k] fp32 final normaliser z_T, or NULL
 *   chunk     chunk length C: 0 = let the library choose, else one of
 *             16, 32, 64, 128 (the result does not depend on it beyond
 *             rounding)
 *   workspace device scratch of at least la_workspace_size(...) bytes
 *             (may be NULL when that size is 0); overwritten by the call
 *   dev_status  device int or NULL (see the conventions above)
 *
 * T == 0 is valid: nothing is written to O and the final state equals the
 * initial one.  B == 0 or H == 0 is a no-op.
 * LA_NONCAUSAL ("Linear attention" box, non-causal form): requires every
 * gamma == 1 and S0 == z0 == NULL, else LA_ERR_UNSUPPORTED; S_out / z_out
 * then receive phi(K)^T V and phi(K)^T 1.
 * Errors: LA_ERR_INVALID_ARG (negative size, d_k/d_v not a multiple of 16
 * in [16, 256], a NULL required pointer, misalignment, gamma outside (0, 1],
 * non-finite or negative eps, an unknown flag, dtype or chunk, workspace
 * too small, O overlapping an input); LA_ERR_UNSUPPORTED; LA_ERR_CUDA.
 */
LA_API la_status la_chunk_fwd(const void* Q, const void* K, const void* V, la_dtype dtype,
                              const float* gamma, int B, int H, int T, int d_k, int d_v,
                              unsigned flags, float eps,
                              const float* S0, const float* z0,
                              void* O, float* S_out, float* z_out,
                              int chunk, void* workspace, size_t workspace_bytes,
                              int* dev_status, la_stream_t stream);

/*
 * One recurrent decode step for every (b, h), updating the state in place:
 * "Recurrent Representation" ("RetNet", bembew) and the decode step of the
 * "Linear attention" page (zerotofrontier 21.2, "Decoding, training, and
 * what each costs"; update first, then read, so the token is in its own sum):
 *
 *   S = gamma S + phi(k) v^T ;  z = gamma z + phi(k)     (z only if normalising)
 *   o = phi(q)^T S  [ / (phi(q)^T z + eps) ]  [ / max(|phi(q)^T z|, 1) ]
 *
 *   q, k   [B][H][d_k] dtype;  v [B][H][d_v] dtype;  o [B][H][d_v] dtype
 *   S      [B][H][d_k][d_v] fp32, read and written in place
 *   z      [B][H][d_k] fp32, in place; required with LA_NORMALIZE or
 *          LA_NORM_FLOOR, else ignored
 *   flags  LA_PHI_ELU1 | LA_NORMALIZE | LA_NORM_FLOOR (LA_NONCAUSAL is
 *          LA_ERR_UNSUPPORTED)
 * Errors: as la_chunk_fwd.
 */
LA_API la_status la_recurrent_step(const void* q, const void* k, const void* v, la_dtype dtype,
                                   const float* gamma, int B, int H, int d_k, int d_v,
                                   unsigned flags, float eps,
                                   float* S, float* z, void* o,
                                   int* dev_status, la_stream_t stream);

/*
 * Chunkwise forward with a per-token (data-dependent) scalar decay in place
 * of the per-head gamma:
 *
 *   S_t = a_t S_{t-1} + phi(k_t) v_t^T,   z_t = a_t z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t  [ normalised as in la_chunk_fwd ]
 *
 * with a_t = exp(log_a[b][h][t]).  The generic "decay the old state, add the
 * new contribution, read out" recurrence of "Linear Attention, RWKV, and
 * RetNet" (temporalbook 13.3, subsection 4 "The Unifying Picture"), whose
 * decay G_t depends on the input in the selective case, with G_t = a_t 1 a
 * scalar per head and token; "Efficient and Sparse Transformers"
 * (temporalbook 12.5, "Gated Linear Attention: Toward Input-Dependent
 * Forgetting") has RetNet as the constant case G_t = gamma 1.  The chunkwise
 * form uses cumulative log-decays inside each chunk instead of powers of
 * gamma (the state between chunks decays by the product of the chunk's a_t).
 *
 *   log_a  DEVICE fp32 [B][H][T], natural log of each decay, finite and <= 0
 *          (a_t in (0, 1]); read only; not checked (device memory)
 *   other arguments as la_chunk_fwd (no gamma); flags as la_chunk_fwd, with
 *          or without LA_GATED; LA_NONCAUSAL is LA_ERR_UNSUPPORTED
 *   workspace: at least la_workspace_size(..., flags | LA_GATED, chunk)
 *          bytes (the tensor-core path always needs some: the per-chunk
 *          cumulative decays)
 * Errors: as la_chunk_fwd; LA_ERR_INVALID_ARG also for log_a == NULL or
 * misaligned when T > 0.
 */
LA_API la_status la_chunk_fwd_gated(const void* Q, const void* K, const void* V,
                                    la_dtype dtype, const float* log_a, int B, int H, int T,
                                    int d_k, int d_v, unsigned flags, float eps,
                                    const float* S0, const float* z0,
                                    void* O, float* S_out, float* z_out,
                                    int chunk, void* workspace, size_t workspace_bytes,
                                    int* dev_status, la_stream_t stream);

/*
 * One decode step with a per-token decay: la_recurrent_step with
 * S = a S + phi(k) v^T, z = a z + phi(k), a = exp(log_a[b][h]).
 *   log_a  DEVICE fp32 [B][H] (this step's decays), finite and <= 0
 * Errors: as la_recurrent_step; LA_ERR_INVALID_ARG also for log_a == NULL or
 * misaligned.
 */
LA_API la_status la_recurrent_step_gated(const void* q, const void* k, const void* v,
                                         la_dtype dtype, const float* log_a, int B, int H,
                                         int d_k, int d_v, unsigned flags, float eps,
                                         float* S, float* z, void* o,
                                         int* dev_status, la_stream_t stream);

/*
 * Backward pass: the gradients of la_chunk_fwd's outputs, for the loss
 *   L = sum_t dO_t . o_t + <dS_T, S_T> + <dz_T, z_T>
 * with respect to Q, K, V and the initial state.  "Linear attention"
 * (zerotofrontier 21.2), "Decoding, training, and what each costs": the
 * gradients are cumulative sums too, forward in time for the queries and
 * backward in time for the keys and values, so no intermediate state is
 * stored (the states are recomputed, chunk by chunk).
 *
 *   Q, K, V, gamma, flags, eps, S0, z0   as the forward call that made O (flags:
 *          LA_PHI_ELU1, LA_NORMALIZE, LA_NORM_FLOOR; LA_NONCAUSAL is
 *          LA_ERR_UNSUPPORTED)
 *   dO     [B][H][T][d_v] dtype: the loss's gradient with respect to O
 *   dS_T   [B][H][d_k][d_v] fp32 or NULL (zero); dz_T [B][H][d_k] fp32 or NULL
 *   dQ, dK [B][H][T][d_k] dtype, dV [B][H][T][d_v] dtype: outputs (may not
 *          overlap any input)
 *   dS0    [B][H][d_k][d_v] fp32 or NULL, dz0 [B][H][d_k] fp32 or NULL: the
 *          initial state's gradients
 *   workspace: at least la_bwd_workspace_size(...) bytes (the sweeps'
 *          segment states and, when normalising, per-token denominators; the
 *          tensor-core passes' operands where they run)
 * d_k and d_v must be at most 128 (LA_ERR_UNSUPPORTED otherwise).  Paths: bf16
 * calls with per-head decay, no normaliser and LA_PHI_ELU1 or no feature map
 * run as three tensor-core forward passes; normalised bf16 calls with per-head decay
 * and d_v = 64 take dq from the CUDA cores in fp32 and dk, dv from two
 * tensor-core passes (dq of the normalised form cancels too much for bf16
 * operands); everything else runs in fp32 on the CUDA cores.
 * LA_PHI_TAYLOR: the Taylor feature map as in la_chunk_fwd (d_k = 16, not with
 * LA_PHI_ELU1, not with per-token decays); S0, z0, dS_T, dz_T, dS0 and dz0 then
 * have 1 + d_k + d_k^2 = 273 rows in the map's order, and dQ, dK are the
 * gradients of the raw 16-wide q and k (through the map's transpose Jacobian).
 * Errors as la_chunk_fwd.
 */
LA_API la_status la_chunk_bwd(const void* Q, const void* K, const void* V, const void* dO,
                              la_dtype dtype, const float* gamma, int B, int H, int T, int d_k,
                              int d_v, unsigned flags, float eps, const float* S0,
                              const float* z0, const float* dS_T, const float* dz_T, void* dQ,
                              void* dK, void* dV, float* dS0, float* dz0, void* workspace,
                              size_t workspace_bytes, int* dev_status, la_stream_t stream);

/* la_chunk_bwd with the per-token decay of la_chunk_fwd_gated (log_a: DEVICE
 * fp32 [B][H][T]) in place of gamma.  The decays themselves get no gradient. */
LA_API la_status la_chunk_bwd_gated(const void* Q, const void* K, const void* V, const void* dO,
                                    la_dtype dtype, const float* log_a, int B, int H, int T,
                                    int d_k, int d_v, unsigned flags, float eps,
                                    const float* S0, const float* z0, const float* dS_T,
                                    const float* dz_T, void* dQ, void* dK, void* dV,
                                    float* dS0, float* dz0, void* workspace,
                                    size_t workspace_bytes, int* dev_status, la_stream_t stream);

/* Bytes of workspace la_chunk_bwd needs (pure host arithmetic; 0 for arguments
 * it would reject). */
LA_API size_t la_bwd_workspace_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype,
                                    unsigned flags);

/*
 * la_chunk_fwd for callers that cannot allocate device memory.  The source
 * pages have no counterpart to this entry point.
 *
 * la_chunk_fwd may need caller-provided scratch (la_workspace_size).  Some
 * callers cannot call cudaMalloc: a plugin inside a host framework that owns
 * every device allocation and passes the plugin only its inputs and outputs,
 * or a serving loop that must not allocate once running (cudaMalloc can
 * synchronise the device and can fail under memory pressure).  This entry
 * point takes the same arguments as la_chunk_fwd minus the workspace and
 * uses instead a fixed scratch array compiled into the library: a file-scope
 * device array of LA_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the
 * library holds until the process exits.  It allocates nothing.
 *
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it.  The cached address holds until the
 *     device is reset (cudaDeviceReset); calls after a reset in the same
 *     process are not supported.
 *   - Calls whose la_workspace_size exceeds LA_NOALLOC_SCRATCH_BYTES return
 *     LA_ERR_INVALID_ARG without launching anything.
 *   - Every call shares the one array, and the array keeps whatever the last
 *     call left in it.  Nothing needs clearing: within a call every scratch
 *     byte is written before it is read (the state walk writes each segment's
 *     contribution, zeros included where no normaliser is carried, before the
 *     scan or the output walk reads it).  Calls that overlap on the GPU
 *     (different streams, or host threads) race on the array and give wrong
 *     results; serialise them.
 *   - Errors otherwise as la_chunk_fwd; LA_ERR_CUDA if the address lookup fails.
 */
#define LA_NOALLOC_SCRATCH_BYTES (16u << 20)
LA_API la_status la_chunk_fwd_noalloc(const void* Q, const void* K, const void* V,
                                      la_dtype dtype, const float* gamma, int B, int H, int T,
                                      int d_k, int d_v, unsigned flags, float eps,
                                      const float* S0, const float* z0,
                                      void* O, float* S_out, float* z_out, int chunk,
                                      int* dev_status, la_stream_t stream);

/*
 * la_chunk_fwd on HOST buffers, the copies included: the end-to-end call for a
 * caller whose inputs and outputs live in host memory (the operation is
 * la_chunk_fwd's; the pages have no counterpart to the copies).
 *
 *   Q, K, V, S0, z0   as la_chunk_fwd, in HOST memory (pinned, e.g. by
 *                     cudaHostAlloc, for the copies to run asynchronously and
 *                     overlap; pageable memory works, with serialised copies)
 *   O, S_out, z_out   as la_chunk_fwd, in HOST memory; written when the call's
 *                     work on `stream` completes
 *   pieces            the batch is cut into `pieces` groups of whole sequences
 *                     (1 <= pieces <= B); piece i is copied in, computed and
 *                     copied out in order on one of two streams the call creates
 *                     (i mod 2), into slot i mod 2 of the arena, so one piece's
 *                     copies overlap another's compute
 *   arena, arena_bytes  caller-owned DEVICE memory of at least
 *                     la_host_arena_size(...) bytes (16-byte aligned): two
 *                     slots of one piece's inputs, outputs and workspace; the
 *                     library allocates nothing
 *   stream            the call's work starts after the work already on `stream`,
 *                     and work enqueued on `stream` afterwards starts after the
 *                     call's (events); the call returns without waiting: the host
 *                     buffers must stay valid, and the outputs are not read, until
 *                     `stream` has passed the call's work
 * gamma and the flags as la_chunk_fwd (the per-token decay is not taken here).
 * Every check of the per-piece calls runs before anything is enqueued.
 * Errors: as la_chunk_fwd; LA_ERR_INVALID_ARG also for pieces outside [1, B],
 * a NULL host input or output when T > 0, or an arena that is too small or
 * misaligned; LA_ERR_CUDA if a copy, stream or event call fails.
 */
LA_API size_t la_host_arena_size(int B, int H, int T, int d_k, int d_v, la_dtype dtype,
                                 unsigned flags, int chunk, int pieces);
LA_API la_status la_chunk_fwd_host(const void* Q, const void* K, const void* V, la_dtype dtype,
                                   const float* gamma, int B, int H, int T, int d_k, int d_v,
                                   unsigned flags, float eps, const float* S0, const float* z0,
                                   void* O, float* S_out, float* z_out, int chunk, int pieces,
                                   void* arena, size_t arena_bytes, int* dev_status,
                                   la_stream_t stream);

/*
 * Test and diagnostic switches (no counterpart on the pages).  Process-wide,
 * all 0 by default; they steer no call unless a test sets them.
 *
 *   LA_OPT_PATH           0: automatic path choice.  1: la_chunk_fwd and
 *                         la_chunk_bwd run on the fp32 CUDA-core kernels
 *                         (la_workspace_size and la_bwd_workspace_size answer
 *                         for that path).  2: la_chunk_fwd runs on the
 *                         tensor-core kernels or answers LA_ERR_UNSUPPORTED.
 *   LA_OPT_TC_LOCKSTEP    1: the tensor-core forward uses its lockstep kernel
 *                         where it would use the pipelined one.
 *   LA_OPT_FORCE_TIMEOUT  1: the tensor-core forward kernels first wait 1 ms on
 *                         a barrier nothing arrives on, then record
 *                         LA_ERR_TIMEOUT in dev_status and return without
 *                         computing (the device status path, exercised with
 *                         neither a hang nor a fault).
 *
 * Returns the option's previous value, or -1 (nothing changed) for an unknown
 * option or an out-of-range value.  Set a switch before enqueuing the calls it
 * should affect; it is read when a call is made, not when its kernels run.
 */
#define LA_OPT_PATH 1
#define LA_OPT_TC_LOCKSTEP 2
#define LA_OPT_FORCE_TIMEOUT 3
LA_API int la_debug_set(int option, int value);

/*
 * Launch tracing (profiling aid; no counterpart on the pages).  While enabled,
 * the library records a pair of CUDA events on the launching stream around
 * every kernel it enqueues, for up to `capacity` launches (capacity <= 0
 * disables tracing and frees the events).  la_trace_collect waits for the
 * recorded launches, writes up to max_records {kernel name, device ms}
 * records (names are static strings) and resets the log; it returns the
 * number written, or -LA_ERR_CUDA.  Not thread-safe across concurrent
 * streams' interleaved calls beyond keeping each record's pair consistent.
 */
typedef struct {
    const char* kernel;
    float ms;
} la_trace_record;

LA_API int la_trace_enable(int capacity);
LA_API int la_trace_collect(la_trace_record* out, int max_records);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
