// Chunkwise forward on the tcgen05 tensor cores (bf16 inputs, fp32
// accumulation), sm_103a.
//
// "Chunked Recurrent Representation" ("RetNet", bembew): chunks of C = 128
// tokens; inside a chunk the parallel form (Q K^T . D) V, across chunks the
// carried state S.  Written out from the recurrence (the pages give the
// chunkwise form only in words), for a chunk of L <= C rows, local indices
// i (query) and j (key), entry state S_{c-1}:
//
//   P_ij = (phi(q_i) . phi(k_j)) gamma^(i-j)   (j <= i, else 0)
//   O_c  = P V_c + (xi . phi(Q_c)) S_{c-1}                 xi_i   = gamma^(i+1)
//   S_c  = gamma^L S_{c-1} + (zeta . phi(K_c))^T V_c       zeta_j = gamma^(L-1-j)
//   normaliser: den_i = sum_j P_ij + xi_i phi(q_i) . z_{c-1} + eps,
//               z_c = gamma^L z_{c-1} + sum_j zeta_j phi(k_j)
//
// One CTA owns one unit: a (b, h) sequence, a block of DVB value columns and
// a segment of consecutive chunks; it walks the chunks in order with S held
// in tensor memory (fp32) the whole time.  Per chunk (all four contractions
// on the tensor cores, M = 128):
//   MMA1  scores = Q K^T            A = Q (K-major smem)   B = K (K-major smem)
//   E1    P = bf16(scores . D)      tcgen05.ld -> mask -> tcgen05.st (P stays in TMEM)
//   E3    S_bf16 = bf16(S) in smem; S = gamma^L S in TMEM
//   MMA2  O = P V                   A = P (TMEM)           B = V (MN-major smem)
//   MMA3  O += Q^ S_bf16            A = Q^ (K-major smem)  B = S_bf16 (MN-major smem)
//   MMA4  S += K^^T V               A = K^ (MN-major smem) B = V (MN-major smem)
//   E2    O -> bf16 -> global
// Q, K, V arrive by TMA (128-byte swizzle) into a two-stage ring, so chunk
// c+1 loads while chunk c computes.  Only non-negative powers of gamma are
// used: small gamma underflows to 0 instead of overflowing.
//
// Unit kinds (one kernel, `mode`):
//   kFull       outputs and state from an entry state (zero, S0 or a segment entry)
//   kStateOnly  only the state walk (MMA4), from zero: a segment's own
//               contribution sum_t gamma^(end-1-t) phi(k_t) v_t^T
//   kNonCausal  gamma = 1: a state walk over the whole sequence, then every
//               chunk reads the final summary (MMA3 only)
//
// Every wait on an mbarrier is bounded by a time limit; on expiry the CTA
// records LA_ERR_TIMEOUT in dev_status, stops issuing work, frees its tensor
// memory and returns.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "chunk_tc_common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"
#include "trace.h"

namespace la {

using namespace tck;

namespace {

constexpr int kThreads = 128;   // 4 warps: warp w owns TMEM lanes 32w .. 32w+31
constexpr uint32_t kColO = 128;   // O accumulator (DVB cols), then the state S (DVB cols)

// TMEM columns: scores/P 128 + O DVB + S DVB, rounded up to a power of two
// (256 for DVB = 64, so two CTAs can share an SM; 512 for DVB = 128).
template <int DVB>
struct Tmem {
    static constexpr uint32_t kColS = kColO + DVB;
    static constexpr uint32_t kCols = (128 + 2 * DVB) <= 256 ? 256 : 512;
};

template <int DK, int DVB>
struct Layout {
    static constexpr uint32_t kQ = (DK / 64) * kBlk;
    static constexpr uint32_t kK = (DK / 64) * kBlk;
    static constexpr uint32_t kV = (DVB / 64) * kBlk;
    static constexpr uint32_t kStage = kQ + kK + kV;
    static constexpr uint32_t kSB = (DVB / 64) * (DK * 128);  // S_bf16, MN-major
    static constexpr uint32_t oSB = 2 * kStage;
    static constexpr uint32_t oZ = oSB + kSB;             // float z[DK]
    static constexpr uint32_t oZP = oZ + DK * 4;          // float colsum partials [256/DK][DK]
    static constexpr uint32_t oBar = oZP + 256 * 4;       // 4 mbarriers
    static constexpr uint32_t oSlot = oBar + 4 * 8;       // TMEM base address
    static constexpr uint32_t kBytes = oSlot + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};

template <int DK, int DVB>
__global__ void __launch_bounds__(kThreads, 1) chunk_tc_kernel(const __grid_constant__ TcParams p) {
    using Lay = Layout<DK, DVB>;
    constexpr uint32_t kColS = Tmem<DVB>::kColS;
    constexpr uint32_t kTmemCols = Tmem<DVB>::kCols;
    extern __shared__ __align__(1024) char smem_raw[];
    char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* zs = reinterpret_cast<float*>(sm + Lay::oZ);
    uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + Lay::oBar);  // [2]
    uint64_t* bar_mma = bar_full + 2;
    uint64_t* bar_never = bar_full + 3;
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Lay::oSlot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int unit = blockIdx.x;
    const int seg = unit % p.n_seg;
    const int dvb = (unit / p.n_seg) % p.n_dvb;
    const int bh = unit / (p.n_seg * p.n_dvb);
    const int h = bh % p.H;
    const int v0 = dvb * DVB;
    const float l2g = p.g.log2g[h];
    const bool unit_gamma = p.g.gamma[h] == 1.0f;
    const int n_chunks = (p.T + kC - 1) / kC;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(n_chunks, c_begin + p.seg_chunks);

    if (tid == 0) {
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_never, 1);
        fence_mbar_init();
        prefetch_tensormap(&p.tmQ);
        prefetch_tensormap(&p.tmK);
        prefetch_tensormap(&p.tmV);
    }
    if (warp == 0) {
        tmem_alloc(slot, kTmemCols);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t sbase = smem_addr(sm);

    bool failed = false;
    if (p.force_timeout) {  // test hook: a wait on a barrier nothing arrives on
        if (tid == 0 && !mbar_wait(bar_never, 0, p.wait_ns)) record_status(p.dev_status, LA_ERR_TIMEOUT);
        failed = true;
    }

    // ---- entry state: S rows d < DK into TMEM lanes, z into shared memory
    if (!failed) {
        const int sidx = bh * p.in_nseg + seg;
        const bool has_in = p.S_in != nullptr && p.mode != kStateOnly && p.mode != kNonCausal;
        for (int c0 = 0; c0 < DVB; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float x = 0.f;
                if (has_in && tid < DK)
                    x = p.S_in[((size_t)sidx * DK + tid) * p.dv + v0 + c0 + e];
                r[e] = __float_as_uint(x);
            }
            tmem_st32(tbase + lane_off + kColS + c0, r);
        }
        tmem_st_wait();
        for (int d = tid; d < DK; d += kThreads)
            zs[d] = (has_in && p.z_in) ? p.z_in[(size_t)sidx * DK + d] : 0.f;
    }

    const uint32_t kBytesQ = Lay::kQ, kBytesK = Lay::kK, kBytesV = Lay::kV;
    const int z3 = bh;
    // Issues the TMA loads of chunk c for walk `w` into stage s.
    auto issue = [&](int c, int s, bool need_q, bool need_kv) {
        char* st = sm + s * Lay::kStage;
        uint32_t bytes = (need_q ? kBytesQ : 0) + (need_kv ? kBytesK + kBytesV : 0);
        mbar_arrive_expect_tx(&bar_full[s], bytes);
        const int y = c * kC;
        if (need_q)
            for (int b = 0; b < DK / 64; ++b) tma_load_3d(st + b * kBlk, &p.tmQ, b * 64, y, z3, &bar_full[s]);
        if (need_kv) {
            for (int b = 0; b < DK / 64; ++b)
                tma_load_3d(st + Lay::kQ + b * kBlk, &p.tmK, b * 64, y, z3, &bar_full[s]);
            for (int b = 0; b < DVB / 64; ++b)
                tma_load_3d(st + Lay::kQ + Lay::kK + b * kBlk, &p.tmV, v0 + b * 64, y, z3, &bar_full[s]);
        }
    };

    uint32_t full_phase[2] = {0, 0};
    uint32_t mma_phase = 0;
    bool inflight[2] = {false, false};  // a TMA fill of the stage not yet waited for
    bool mma_inflight = false;          // MMAs committed but not yet waited for
    // walk 0: the causal walk (or the state walk of kStateOnly / kNonCausal);
    // walk 1: the non-causal read-out walk.
    const int n_walks = p.mode == kNonCausal ? 2 : 1;
    for (int walk = 0; walk < n_walks && !failed; ++walk) {
        const bool do_out = (p.mode == kFull) || (p.mode == kNonCausal && walk == 1);
        const bool do_intra = p.mode == kFull;
        const bool do_state = (p.mode == kFull) || (p.mode == kStateOnly) ||
                              (p.mode == kNonCausal && walk == 0);
        const bool need_q = do_out;
        const bool need_kv = do_intra || do_state;
        const int cb = p.mode == kNonCausal ? 0 : c_begin;
        const int ce = p.mode == kNonCausal ? n_chunks : c_end;

        if (p.mode == kNonCausal && walk == 1) {
            // the summary is final: one bf16 copy of S for every read-out MMA
            if (tid < DK) {
                for (int c0 = 0; c0 < DVB; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColS + c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e8 = 0; e8 < 32; e8 += 8) {
                        const int v = c0 + e8;
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[e8 + 0]), __uint_as_float(r[e8 + 1]));
                        w.y = pack_bf16x2(__uint_as_float(r[e8 + 2]), __uint_as_float(r[e8 + 3]));
                        w.z = pack_bf16x2(__uint_as_float(r[e8 + 4]), __uint_as_float(r[e8 + 5]));
                        w.w = pack_bf16x2(__uint_as_float(r[e8 + 6]), __uint_as_float(r[e8 + 7]));
                        *reinterpret_cast<uint4*>(sm + Lay::oSB + (v >> 6) * (DK * 128) +
                                                  sw128_offset(tid, v & 63)) = w;
                    }
                }
            } else {
                for (int c0 = 0; c0 < DVB; c0 += 32) {  // keep the warp-wide ld collective
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColS + c0, r);
                    tmem_ld_wait();
                }
            }
            fence_proxy_async_smem();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
        }
        if (cb >= ce) continue;
        if (tid == 0) issue(cb, 0, need_q, need_kv);
        inflight[0] = true;

        for (int c = cb; c < ce; ++c) {
            const int it = c - cb;
            const int s = it & 1;
            char* st = sm + s * Lay::kStage;
            char* tQ = st;
            char* tK = st + Lay::kQ;
            const int L = min(kC, p.T - c * kC);
            if (c + 1 < ce) {
                if (tid == 0) issue(c + 1, s ^ 1, need_q, need_kv);
                inflight[s ^ 1] = true;
            }

            bool to = !mbar_wait(&bar_full[s], full_phase[s], p.wait_ns);
            if (__syncthreads_or(to)) {
                failed = true;
                break;
            }
            full_phase[s] ^= 1;
            inflight[s] = false;
            // phi on q and k (rows >= L zeroed: phi(0) = 1 must not leak in)
            if (p.phi) {
                if (need_q) row_pass(tQ, DK / 64, true, [&](int r) { return r < L ? 1.f : 0.f; }, tid, kThreads);
                if (need_kv) row_pass(tK, DK / 64, true, [&](int r) { return r < L ? 1.f : 0.f; }, tid, kThreads);
                fence_proxy_async_smem();
            }
            fence_before_sync();
            __syncthreads();
            fence_after_sync();

            float r_i = 0.f;  // row sum of the scores (normaliser)
            if (do_intra) {
                if (tid == 0) {
                    // MMA1: scores[128 x 128] = Q K^T, K = DK
                    const uint32_t id = idesc_bf16(128, 128, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
                        mma_ss(tbase + kColP, smem_desc_sw128(sbase + (uint32_t)(tQ - sm) + off, 16, 1024),
                               smem_desc_sw128(sbase + (uint32_t)(tK - sm) + off, 16, 1024), id, kk > 0);
                    }
                    mma_commit(bar_mma);
                }
                mma_inflight = true;
                to = !mbar_wait(bar_mma, mma_phase, p.wait_ns);
                if (__syncthreads_or(to)) {
                    failed = true;
                    break;
                }
                mma_phase ^= 1;
                mma_inflight = false;
                fence_after_sync();
                // E1: row i = tid: P_ij = s_ij gamma^(i-j) for j <= i, packed bf16 back into TMEM
                const int i = tid;
                const float gam = p.g.gamma[h];
#pragma unroll
                for (int c0 = 0; c0 < kC; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColP + c0, r);
                    tmem_ld_wait();
                    uint32_t pk[16];
                    // gamma^(i-j) by a running product from the piece's top column down
                    const int jt = min(i, c0 + 31);
                    float w = (unit_gamma || jt < c0) ? 1.f : gamma_pow(l2g, (float)(i - jt));
                    float a[32];
#pragma unroll
                    for (int e = 31; e >= 0; --e) {
                        float x = 0.f;
                        if (c0 + e <= i) {
                            x = __uint_as_float(r[e]);
                            if (!unit_gamma) {
                                x *= w;
                                w *= gam;
                            }
                        }
                        a[e] = x;
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        pk[e >> 1] = pack_bf16x2(a[e], a[e + 1]);
                        // the row sum in fp32, before P is rounded: with signed features
                        // the denominator can be a small difference of large sums
                        r_i += a[e] + a[e + 1];
                    }
                    tmem_st16(tbase + lane_off + kColP + (c0 >> 1), pk);
                }
                tmem_st_wait();
            }
            // the normaliser state's sum_j zeta_j phi(K)[j], in fp32 from the tile before
            // it is scaled (added to z below, after z_{c-1} has been read)
            float* zpart = reinterpret_cast<float*>(sm + Lay::oZP);
            if (p.track_z && do_state) {
                if (unit_gamma)
                    colsum_partial<DK>(tK, tid, zpart);
                else
                    colsum_partial_decayed<DK>(tK, tid, zpart, L, l2g, p.g.gamma[h]);
            }
            // normaliser: qz_i = xi_i (q^_i . z_{c-1}), in fp32 from the unscaled tile (with
            // signed features q . z can be a small difference of large terms)
            float qz = 0.f;
            if (p.normalize && do_out) {
                const int i = tid;
#pragma unroll 4
                for (int d8 = 0; d8 < DK; d8 += 8) {
                    const uint4 u = *reinterpret_cast<const uint4*>(tQ + (d8 >> 6) * kBlk + sw128_offset(i, d8 & 63));
                    const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(hq[e]);
                        qz = fmaf(x.x, zs[d8 + 2 * e], qz);
                        qz = fmaf(x.y, zs[d8 + 2 * e + 1], qz);
                    }
                }
                if (!unit_gamma) qz *= gamma_pow(l2g, (float)(i + 1));
            }
            // Q^ = xi . Q, K^ = zeta . K (rows >= L of K get 0), once every read above is done
            const float gL = unit_gamma ? 1.f : gamma_pow(l2g, (float)L);
            if (!unit_gamma || (p.track_z && do_state)) __syncthreads();
            if (!unit_gamma) {
                if (do_out)
                    row_pass(tQ, DK / 64, false, [&](int r) { return gamma_pow(l2g, (float)(r + 1)); },
                             tid, kThreads);
                if (do_state)
                    row_pass(tK, DK / 64, false,
                             [&](int r) { return r < L ? gamma_pow(l2g, (float)(L - 1 - r)) : 0.f; },
                             tid, kThreads);
            }
            __syncthreads();
            // E3: S_bf16 = bf16(S_{c-1}) (for MMA3), S = gamma^L S (before MMA4 accumulates)
            const bool need_sb = do_out && p.mode == kFull;
            const bool scale_s = do_state && !unit_gamma;
            if (need_sb || scale_s) {
                for (int c0 = 0; c0 < DVB; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColS + c0, r);
                    tmem_ld_wait();
                    if (need_sb && tid < DK) {
#pragma unroll
                        for (int e8 = 0; e8 < 32; e8 += 8) {
                            const int v = c0 + e8;
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(r[e8 + 0]), __uint_as_float(r[e8 + 1]));
                            w.y = pack_bf16x2(__uint_as_float(r[e8 + 2]), __uint_as_float(r[e8 + 3]));
                            w.z = pack_bf16x2(__uint_as_float(r[e8 + 4]), __uint_as_float(r[e8 + 5]));
                            w.w = pack_bf16x2(__uint_as_float(r[e8 + 6]), __uint_as_float(r[e8 + 7]));
                            *reinterpret_cast<uint4*>(sm + Lay::oSB + (v >> 6) * (DK * 128) +
                                                      sw128_offset(tid, v & 63)) = w;
                        }
                    }
                    if (scale_s) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * gL);
                        tmem_st32(tbase + lane_off + kColS + c0, r);
                    }
                }
                if (scale_s) tmem_st_wait();
            }
            fence_proxy_async_smem();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();

            // MMA2..4
            if (tid == 0) {
                const uint32_t vbase = sbase + (uint32_t)(tK - sm) + Lay::kK;
                if (do_intra) {  // MMA2: O = P V, K = 128 tokens
                    const uint32_t id = idesc_bf16(128, DVB, 0, 1);
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_ts(tbase + kColO, tbase + kColP + kk * 8,
                               smem_desc_sw128(vbase + kk * 2048, kBlk, 1024), id, kk > 0);
                }
                if (do_out) {  // MMA3: O (+)= Q^ S_bf16, K = DK
                    const uint32_t id = idesc_bf16(128, DVB, 0, 1);
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t offa = (kk >> 2) * kBlk + (kk & 3) * 32;
                        mma_ss(tbase + kColO, smem_desc_sw128(sbase + (uint32_t)(tQ - sm) + offa, 16, 1024),
                               smem_desc_sw128(sbase + Lay::oSB + kk * 2048, DK * 128, 1024), id,
                               (do_intra || kk > 0) ? 1u : 0u);
                    }
                }
                if (do_state) {  // MMA4: S += K^^T V, M = 128 (rows >= DK unused), K = 128 tokens
                    const uint32_t id = idesc_bf16(128, DVB, 1, 1);
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_ss(tbase + kColS, smem_desc_sw128(sbase + (uint32_t)(tK - sm) + kk * 2048, kBlk, 1024),
                               smem_desc_sw128(vbase + kk * 2048, kBlk, 1024), id, 1u);
                }
                mma_commit(bar_mma);
            }
            mma_inflight = true;
            // normaliser state: z_c = gamma^L z + sum_j zeta_j phi(K)[j]   (z_{c-1} already
            // used above; the partial sums were taken before the scaling)
            if (p.track_z && do_state) {
                if (tid < DK) zs[tid] = fmaf(unit_gamma ? 1.f : gL, zs[tid], colsum_total<DK>(zpart, tid));
            }
            to = !mbar_wait(bar_mma, mma_phase, p.wait_ns);
            if (__syncthreads_or(to)) {
                failed = true;
                break;
            }
            mma_phase ^= 1;
            mma_inflight = false;
            fence_after_sync();
            // E2: O row i = tid -> global (rows < L)
            if (do_out) {
                const int i = tid;
                const float inv = p.normalize ? 1.f / norm_den(r_i + qz, p.normalize, p.eps) : 1.f;
                __nv_bfloat16* orow = p.O + ((size_t)bh * p.T + (size_t)c * kC + i) * p.dv + v0;
                for (int c0 = 0; c0 < DVB; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColO + c0, r);
                    tmem_ld_wait();
                    if (i < L) {
#pragma unroll
                        for (int e8 = 0; e8 < 32; e8 += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(r[e8 + 0]) * inv, __uint_as_float(r[e8 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(r[e8 + 2]) * inv, __uint_as_float(r[e8 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(r[e8 + 4]) * inv, __uint_as_float(r[e8 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(r[e8 + 6]) * inv, __uint_as_float(r[e8 + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + c0 + e8) = w;
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            fence_before_sync();
            __syncthreads();  // stage s may be refilled by the next iteration's TMA
            fence_after_sync();
        }
    }

    // ---- exit state
    if (!failed && p.S_out) {
        const bool write = !p.out_last_only || seg == p.n_seg - 1;
        const int oidx = bh * p.out_nseg + (p.out_last_only ? 0 : seg);
        for (int c0 = 0; c0 < DVB; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tbase + lane_off + kColS + c0, r);
            tmem_ld_wait();
            if (write && tid < DK) {
                float* srow = p.S_out + ((size_t)oidx * DK + tid) * p.dv + v0 + c0;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(srow + e) =
                        make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                    __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
            }
        }
        if (write && p.z_out && dvb == 0)
            for (int d = tid; d < DK; d += kThreads) p.z_out[(size_t)oidx * DK + d] = zs[d];
    }
    if (failed) {
        record_status(p.dev_status, LA_ERR_TIMEOUT);
        // let our own copies and MMAs land (bounded) before the memory is released
        if (tid == 0) {
            for (int q = 0; q < 2; ++q)
                if (inflight[q]) mbar_wait(&bar_full[q], full_phase[q], p.wait_ns);
            if (mma_inflight) mbar_wait(bar_mma, mma_phase, p.wait_ns);
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}


template <int DK, int DVB>
cudaError_t launch_tc(const TcParams& prm, int grid, cudaStream_t s) {
    using Lay = Layout<DK, DVB>;
    auto kern = chunk_tc_kernel<DK, DVB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::kAlloc);
    if (e != cudaSuccess) return e;
    static const char* const names[3] = {"chunk_tc_kernel/full", "chunk_tc_kernel/state",
                                         "chunk_tc_kernel/noncausal"};
    TraceScope trace(names[prm.mode], s);
    kern<<<grid, kThreads, Lay::kAlloc, s>>>(prm);
    return cudaGetLastError();
}

}  // namespace

bool tc_ws_supported(int mode, int dk, int dvb, bool normalize);
cudaError_t launch_chunk_tc_ws(int dk, int dvb, bool normalize, const TcParams& prm, int grid,
                               cudaStream_t s, bool pdl);

namespace {

// pdl: the pipelined kernel may be launched as a programmatic dependent of the
// previous kernel (it waits for it before reading entry states); the lockstep
// kernel is always launched in plain stream order.
cudaError_t launch_tc_dispatch(int dk, int dvb, const TcParams& prm, int grid, cudaStream_t s,
                               bool pdl = false) {
    if (grid <= 0) return cudaSuccess;
    if (tc_ws_supported(prm.mode, dk, dvb, prm.normalize != 0))
        return launch_chunk_tc_ws(dk, dvb, prm.normalize != 0, prm, grid, s, pdl);
    if (prm.gate) return cudaErrorInvalidValue;  // the per-token decay runs in the pipelined kernel only
    if (dk == 64 && dvb == 64) return launch_tc<64, 64>(prm, grid, s);
    if (dk == 64 && dvb == 128) return launch_tc<64, 128>(prm, grid, s);
    if (dk == 128 && dvb == 64) return launch_tc<128, 64>(prm, grid, s);
    if (dk == 128 && dvb == 128) return launch_tc<128, 128>(prm, grid, s);
    return cudaErrorInvalidValue;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// Segments per sequence: as many as fit the SMs in one wave (the kernels run
// one CTA per SM), when that is at least two and each segment keeps two or
// more chunks.
int choose_segments(int units, int n_chunks) {
    const int sms = sm_count();
    int P = sms / units;
    if (P > n_chunks / 2) P = n_chunks / 2;
    return P < 2 ? 1 : P;
}

// Entry state of every segment from the segments' own contributions:
//   entry_0 = S0 (or 0),  entry_{q+1} = gamma^len entry_q + agg_q
// (len = the common segment length).  One thread per state element; z rides
// along on the threads of column 0.  The contributions are loaded in batches
// of kScanBatch before the recurrence runs over them, so a thread waits for
// memory once per batch rather than once per segment.  Launched as a
// programmatic dependent of the state walk: it lets the output walk be
// scheduled at once and waits for the state walk's results.
// With the per-token decay the decay over segment q is 2^(seg_l2[bh][q]), the
// segment's total log2 decay that the state walk wrote.
constexpr int kScanBatch = 8;
__global__ void segment_scan_kernel(const float* __restrict__ S0, const float* __restrict__ z0,
                                    const float* __restrict__ agg, const float* __restrict__ zagg,
                                    float* __restrict__ entry, float* __restrict__ zentry,
                                    size_t total, int H, int P, int seg_len, int dk, int dv,
                                    const float* __restrict__ seg_l2,
                                    const __grid_constant__ KernelGammas g) {
    tc::griddep_launch_dependents();
    tc::griddep_wait();
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const size_t per = (size_t)dk * dv;
    const size_t bh = idx / per;
    const size_t e = idx % per;
    const float gseg = seg_l2 ? 0.f : gamma_pow(g.log2g[bh % H], (float)seg_len);
    float x = S0 ? S0[bh * per + e] : 0.f;
    const bool do_z = (e % dv) == 0;
    const size_t d = e / dv;
    float zz = (do_z && z0) ? z0[bh * dk + d] : 0.f;
    for (int q0 = 0; q0 < P; q0 += kScanBatch) {
        float a[kScanBatch], za[kScanBatch], gq[kScanBatch];
#pragma unroll
        for (int b = 0; b < kScanBatch; ++b) {  // the last segment's contribution is not needed
            const int q = q0 + b;
            a[b] = q + 1 < P ? agg[(bh * P + q) * per + e] : 0.f;
            za[b] = (do_z && zagg && q + 1 < P) ? zagg[(bh * P + q) * dk + d] : 0.f;
            gq[b] = seg_l2 ? (q + 1 < P ? exp2f(seg_l2[bh * P + q]) : 0.f) : gseg;
        }
#pragma unroll
        for (int b = 0; b < kScanBatch; ++b) {
            const int q = q0 + b;
            if (q >= P) break;
            entry[(bh * P + q) * per + e] = x;
            if (do_z) zentry[(bh * P + q) * dk + d] = zz;
            x = fmaf(gq[b], x, a[b]);
            if (do_z) zz = fmaf(gq[b], zz, za[b]);
        }
    }
}

// Per chunk of every sequence, for the per-token decay: the cumulative log2
// decays b_i = sum_{s<=i} log2 a_s inside the chunk (flat past the end of the
// sequence) and the decays a_i themselves, into gate[bh][c][0..127] and
// [128..255].  One warp per chunk: each lane scans four tokens, then the lanes'
// totals are scanned with shuffles.
// It also flags each chunk whose decay from its first row to its last is below
// 2^-160, or not a number (flags[bh][c] = 1): the factored build's factors about the
// chunk's middle exponent reach 2^(+-Delta/2) for a decay of 2^-Delta, and past 2^80
// products of them with the data would leave the bf16 range, so the chunk's CTA takes
// the build with row scalings.
__global__ void gate_prep_kernel(const float* __restrict__ log_a, float* __restrict__ gate, int T,
                                 int n_chunks, size_t total_chunks, int* __restrict__ flags) {
    const size_t wid = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= total_chunks) return;  // whole warps only: the block size is a multiple of 32
    const size_t bh = wid / (size_t)n_chunks;
    const int c = (int)(wid % (size_t)n_chunks);
    float l[4], a[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int t = c * kC + lane * 4 + e;
        l[e] = t < T ? log_a[bh * T + t] * 1.44269504088896341f : 0.f;
        a[e] = exp2f(l[e]);
    }
    l[1] += l[0];
    l[2] += l[1];
    l[3] += l[2];
    float inc = l[3];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    const float ex = inc - l[3];  // the lanes before this one
    float* gp = gate + wid * 256;
    reinterpret_cast<float4*>(gp)[lane] = make_float4(l[0] + ex, l[1] + ex, l[2] + ex, l[3] + ex);
    reinterpret_cast<float4*>(gp + 128)[lane] = make_float4(a[0], a[1], a[2], a[3]);
    if (flags) {  // b_0 - b_(L-1): the sum of lanes' totals past token 0 (rows past T add 0)
        const float total = __shfl_sync(0xffffffffu, inc, 31);
        const float first = __shfl_sync(0xffffffffu, l[0], 0);
        if (lane == 0) flags[wid] = (first - total) <= 160.f ? 0 : 1;
    }
}

}  // namespace

namespace tck {
bool make_map_box(CUtensorMap* m, const void* base, int BH, int T, int d, int box_x, bool swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
bool make_map(CUtensorMap* m, const void* base, int BH, int T, int d) {
    return make_map_box(m, base, BH, T, d, 64, true);
}
// [BH][T] rows of `cols` bf16 columns, `pitch` elements apart (a multiple of 8);
// boxes of 64 columns past `cols` read zeros.
bool make_map_pitch(CUtensorMap* m, const void* base, int BH, int T, int cols, int pitch) {
    auto fn = encode_fn();
    if (!fn || pitch % 8 != 0 || cols > pitch) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)pitch * 2, (cuuint64_t)T * pitch * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
bool tc_arch_ok() {
    if (!encode_fn()) return false;
    int dev = 0, major = 0, minor = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}
}  // namespace tck

static int tc_dvb(const ChunkArgs& a);

bool tc_supported(const ChunkArgs& a) {
    if (!a.bf16) return false;
    if (a.dk != 64 && a.dk != 128) return false;
    if (a.dv != 64 && a.dv != 128 && a.dv != 256) return false;
    if (a.chunk != 0 && a.chunk != kC) return false;
    // the per-token decay: causal, in the pipelined kernel only
    if (a.log_a && (a.noncausal || !tc_ws_supported(kFull, a.dk, tc_dvb(a), a.normalize)))
        return false;
    if (a.taylor) return false;  // the Taylor feature map has a kernel of its own
    return tck::tc_arch_ok();
}

// Value columns per CTA: 64 or 128.  With the per-token decay 64 when
// normalising (the pipelined kernel's normalising width) or for d_k = 128 (a
// 128 x 128 stage leaves no shared memory for the chunk's decays).
static int tc_dvb(const ChunkArgs& a) {
    if (a.log_a && (a.normalize || a.dk == 128)) return 64;
    return a.dv == 64 ? 64 : 128;
}

// Reversed time runs in the pipelined kernel's factored-decay build: plain
// retention (no feature map, no normaliser, no z), causal, every head's gamma in
// (0, 1] with gamma^(C-1) >= 2^-64 (gamma = 1 included: the factors are then 1).
bool tc_reverse_supported(const ChunkArgs& a, const KernelGammas& g) {
    if (!tc_supported(a) || a.phi || a.normalize || a.log_a || a.noncausal || a.taylor || a.z_out)
        return false;
    if (a.H <= 0 || a.H > kMaxHeads) return false;
    for (int h = 0; h < a.H; ++h)
        if (!(g.gamma[h] > 0.f && g.gamma[h] <= 1.f && g.log2g[h] * (float)(kC - 1) >= -64.f)) return false;
    return tc_ws_supported(kFull, a.dk, tc_dvb(a), false) && tc_ws_supported(kStateOnly, a.dk, tc_dvb(a), false);
}

// Whether the output walk folds the segments' contributions into its entry states
// itself (no scan kernel): few segments per sequence, and the pipelined kernel runs.
static bool fold_segments(int P, int dk, int dvb, bool normalize) {
    return P <= kFoldMax && tc_ws_supported(kFull, dk, dvb, normalize);
}

namespace {

// The segment plan and the workspace layout of one tensor-core call.
struct TcPlan {
    int n_chunks, units, dvb;
    int P;           // segments per sequence chosen (1: no segments)
    int seg_chunks;  // chunks per segment
    int Pu;          // segments actually used
    // workspace byte offsets: per-token decays per chunk, segment decays, then the
    // segment states (agg, entry: [BH][Pu][dk][dv]; zagg, zentry: [BH][Pu][dk])
    size_t o_gate, o_segl2, o_gflag, o_agg, o_entry, o_zagg, o_zentry, bytes;
};

TcPlan tc_plan(const ChunkArgs& a) {
    TcPlan pl;
    std::memset(&pl, 0, sizeof(pl));
    pl.n_chunks = (a.T + kC - 1) / kC;
    pl.dvb = tc_dvb(a);
    pl.units = a.B * a.H * (a.dv / pl.dvb);
    pl.P = a.noncausal || a.T <= 0 ? 1 : choose_segments(pl.units, pl.n_chunks);
    pl.seg_chunks = pl.P > 1 ? (pl.n_chunks + pl.P - 1) / pl.P : pl.n_chunks;
    pl.Pu = pl.P > 1 ? (pl.n_chunks + pl.seg_chunks - 1) / pl.seg_chunks : 1;
    const size_t nbh = (size_t)a.B * a.H;
    size_t off = 0;
    if (a.log_a && !a.noncausal && a.T > 0) {
        pl.o_gate = off;
        off += nbh * pl.n_chunks * 256 * sizeof(float);
        pl.o_segl2 = off;
        if (pl.P > 1) off += (nbh * pl.P * sizeof(float) + 15) / 16 * 16;
        pl.o_gflag = off;  // per chunk: the factored build does not apply
        off += (nbh * pl.n_chunks * sizeof(int) + 15) / 16 * 16;
    }
    if (pl.P > 1) {
        const size_t st = nbh * pl.P * a.dk * a.dv * sizeof(float), zt = nbh * pl.P * a.dk * sizeof(float);
        pl.o_agg = off;
        pl.o_entry = off + st;
        pl.o_zagg = off + 2 * st;
        pl.o_zentry = off + 2 * st + zt;
        off += 2 * st + 2 * zt;
    }
    pl.bytes = off;
    return pl;
}

}  // namespace

int tc_launch_count(const ChunkArgs& a) {
    if (a.noncausal || a.T <= 0) return 1;
    const TcPlan pl = tc_plan(a);
    const int prep = a.log_a ? 1 : 0;
    if (pl.P <= 1) return 1 + prep;
    return (fold_segments(pl.Pu, a.dk, pl.dvb, a.normalize) ? 2 : 3) + prep;
}

size_t tc_workspace_bytes(const ChunkArgs& a) { return tc_plan(a).bytes; }

void tc_segments(const ChunkArgs& a, int* n_seg, int* seg_chunks) {
    const TcPlan pl = tc_plan(a);
    *n_seg = pl.P > 1 ? pl.Pu : 1;
    *seg_chunks = pl.seg_chunks;
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s,
                            int* launches) {
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int BH = a.B * a.H;
    const int qk_cols = a.qk_cols ? a.qk_cols : a.dk;
    const int qk_pitch = a.qk_pitch ? a.qk_pitch : qk_cols;
    const int v_pitch = a.v_pitch ? a.v_pitch : a.dv;
    if (qk_cols > a.dk || ((a.qk_cols || a.qk_pitch || a.v_pitch) && !tc_ws_supported(kFull, a.dk, tc_dvb(a), a.normalize)))
        return cudaErrorInvalidValue;
    if (!make_map_pitch(&prm.tmQ, a.Q, BH, a.T, qk_cols, qk_pitch) ||
        !make_map_pitch(&prm.tmK, a.K, BH, a.T, qk_cols, qk_pitch) ||
        !make_map_pitch(&prm.tmV, a.V, BH, a.T, a.dv, v_pitch))
        return cudaErrorInvalidValue;
    const TcPlan pl = tc_plan(a);
    if (a.workspace_bytes < pl.bytes || (pl.bytes > 0 && !a.workspace)) return cudaErrorInvalidValue;
    char* ws = static_cast<char*>(a.workspace);
    const int dvb = pl.dvb;
    prm.O = (__nv_bfloat16*)a.O;
    prm.H = a.H;
    prm.T = a.T;
    prm.dv = a.dv;
    prm.n_dvb = a.dv / dvb;
    prm.normalize = norm_mode(a.normalize, a.floor_norm);
    prm.track_z = a.normalize || a.z_out != nullptr;
    prm.phi = a.phi;
    prm.eps = a.eps;
    prm.dev_status = a.dev_status;
    prm.wait_ns = 2000000000ull;
    if (opt_force_timeout()) {
        prm.force_timeout = 1;
        prm.wait_ns = 1000000ull;  // 1 ms
    }
    prm.g = g;
    prm.o_align32 = (reinterpret_cast<uintptr_t>(a.O) & 31u) == 0;
    prm.fact = !a.log_a && !a.phi && !prm.track_z;
    for (int h = 0; h < a.H && prm.fact; ++h)
        prm.fact = g.gamma[h] < 1.f && g.log2g[h] * (float)(kC - 1) >= -64.f;
    if (a.reverse) {  // the factored build alone walks reversed time
        if (!tc_reverse_supported(a, g)) return cudaErrorInvalidValue;
        prm.fact = 1;
        prm.rev = 1;
    }
    const int n_chunks = pl.n_chunks;
    const int units = pl.units;
    *launches = 0;

    if (a.noncausal) {
        prm.mode = kNonCausal;
        prm.seg_chunks = n_chunks;
        prm.n_seg = 1;
        prm.in_nseg = 1;
        prm.S_out = a.S_out;
        prm.z_out = a.z_out;
        prm.out_nseg = 1;
        prm.out_last_only = 1;
        *launches = 1;
        return launch_tc_dispatch(a.dk, dvb, prm, units, s);
    }
    if (a.log_a) {
        // per-token decay: the chunks' cumulative decays first (plain stream order:
        // every later kernel's producer reads them from its first chunk on)
        float* gate = reinterpret_cast<float*>(ws + pl.o_gate);
        const size_t total_chunks = (size_t)BH * n_chunks;
        {
            TraceScope trace("gate_prep_kernel", s);
            gate_prep_kernel<<<(unsigned)((total_chunks * 32 + 255) / 256), 256, 0, s>>>(
                a.log_a, gate, a.T, n_chunks, total_chunks, reinterpret_cast<int*>(ws + pl.o_gflag));
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        prm.gate = gate;
        prm.seg_l2 = pl.P > 1 ? reinterpret_cast<float*>(ws + pl.o_segl2) : nullptr;
        prm.gate_flags = reinterpret_cast<const int*>(ws + pl.o_gflag);
        *launches = 1;
    }
    // The per-token decay without normaliser or z in the factored build wherever a
    // unit's chunks allow it (gate_prep_kernel's flags): the output walk's CTAs pick
    // the factored build or the row scalings each for itself.  A state walk has no
    // row factors and keeps the row scalings.
    const bool pick = a.log_a && !a.phi && !prm.track_z && !a.noncausal && (a.dk == 64 || dvb == 64) &&
                      tc_ws_supported(kFull, a.dk, dvb, false);
    auto dispatch = [&](const TcParams& pp, int grid, bool pdl) -> cudaError_t {
        *launches += 1;
        if (!pick || pp.mode != kFull) return launch_tc_dispatch(a.dk, dvb, pp, grid, s, pdl);
        TcParams p1 = pp;
        p1.fact = 1;  // (the pick kernel)
        return launch_tc_dispatch(a.dk, dvb, p1, grid, s, pdl);
    };
    if (pl.P <= 1) {
        prm.mode = kFull;
        prm.seg_chunks = n_chunks;
        prm.n_seg = 1;
        prm.S_in = a.S0;
        prm.z_in = a.z0;
        prm.in_nseg = 1;
        prm.S_out = a.S_out;
        prm.z_out = a.z_out;
        prm.out_nseg = 1;
        prm.out_last_only = 1;
        return dispatch(prm, units, false);
    }
    // segmented: (1) each segment's own state, (2) scan to entry states, (3) outputs
    const int seg_chunks = pl.seg_chunks;
    const int Pu = pl.Pu;  // segments actually used
    const size_t nbh = (size_t)BH;
    float* agg = a.agg ? a.agg : reinterpret_cast<float*>(ws + pl.o_agg);
    float* entry = reinterpret_cast<float*>(ws + pl.o_entry);
    // (contributions handed in carry no z: nothing reads zagg then)
    float* zagg = a.agg_ready ? nullptr : reinterpret_cast<float*>(ws + pl.o_zagg);
    if (a.agg_ready && (prm.track_z || a.log_a || !a.agg)) return cudaErrorInvalidValue;
    float* zentry = reinterpret_cast<float*>(ws + pl.o_zentry);

    TcParams pa = prm;  // state-only walks of segments 0 .. Pu-2 (the last one's is not needed)
    pa.mode = kStateOnly;
    pa.seg_chunks = seg_chunks;
    pa.n_seg = Pu - 1;
    pa.S_out = agg;
    pa.z_out = zagg;
    pa.out_nseg = Pu;  // contributions keep the [BH][Pu] layout the scan and the fold read
    pa.out_last_only = 0;
    cudaError_t e = a.agg_ready ? cudaSuccess : dispatch(pa, units * (Pu - 1), false);
    if (e != cudaSuccess) return e;
    TcParams pc = prm;
    pc.mode = kFull;
    pc.seg_chunks = seg_chunks;
    pc.n_seg = Pu;
    pc.in_nseg = Pu;
    pc.S_out = a.S_out;
    pc.z_out = a.z_out;
    pc.out_nseg = 1;
    pc.out_last_only = 1;
    if (fold_segments(Pu, a.dk, dvb, a.normalize != 0)) {
        // few segments: the output walk folds the contributions into its entry states
        pc.S_in = agg;
        pc.z_in = zagg;
        pc.in_agg = 1;
        pc.S0 = a.S0;
        pc.z0 = a.z0;
        return dispatch(pc, units * Pu, /*pdl=*/true);
    }
    const size_t total = nbh * (size_t)a.dk * a.dv;
    {
        TraceScope trace("segment_scan_kernel", s);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((total + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, segment_scan_kernel, a.S0, a.z0, (const float*)agg,
                               (const float*)zagg, entry, zentry, total, a.H, Pu, seg_chunks * kC,
                               a.dk, a.dv, (const float*)prm.seg_l2, g);
    }
    if (e != cudaSuccess) return e;
    pc.S_in = entry;
    pc.z_in = zentry;
    *launches += 1;  // the scan
    return dispatch(pc, units * Pu, /*pdl=*/true);
}

}  // namespace la
