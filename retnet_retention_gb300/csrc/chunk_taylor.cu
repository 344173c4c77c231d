// Causal linear attention with the second-order Taylor feature map on the
// tensor cores.
//
// "Linear attention" (zerotofrontier 21.2), section "A Taylor feature map":
// phi(x) = (1, x, vec(x x^T)/sqrt 2) has 1 + d + d^2 entries and
// phi(q)^T phi(k) = 1 + s + s^2/2 with s = q^T k; Based projects q and k to
// d = 16 first, so d_phi = 273.  The queries and keys enter here at their width
// of 16 (32 bytes a token, not 546): the CTA builds the features on chip.
//
// vec(x x^T) is symmetric, so the kernel keeps one feature per unordered pair:
// x_a x_b for a < b and x_a^2 / sqrt 2 for a = b (136 features), then x and 1 —
// 153 features whose dot products are the same 1 + s + s^2/2.  The state in
// these coordinates is the symmetric part of the page's state (rows (a, b) and
// (b, a) summed over sqrt 2); the antisymmetric part of an initial state never
// changes but by the decay (every update k k^T is symmetric), so the final state
// in the page's order is rebuilt exactly from the two.
//
// Per chunk of 128 tokens and block of 64 value columns, with xi_i = gamma^(i+1),
// zeta_j = gamma^(L-1-j) (the forms of the per-head kernels):
//   MMA1  s = q k^T                         (K = 16, the raw q and k)
//   E1    P_ij = (1 + s + s^2/2) gamma^(i-j) for j <= i        (bf16, in TMEM)
//   MMA3  O  = (xi . phi(Q)) S_bf16                            (K = 160 feature columns)
//   MMA4  S^T += [V | 1]^T (zeta . phi(K))                     (z rides as the row of the 1)
//   MMA2  O += P [V | 1]                                       (row sums in column 64)
//   E2    o_i = O_i / (O_i,64 + O_i,65) with the normaliser, else O_i
//   E3    S_bf16 <- S (z as a bf16 value and its residual), S^T *= gamma^L(next chunk)
// The state is held transposed in TMEM (lanes 0..63 the value columns, lane 64
// z, 160 feature columns), so each TMEM lane is one row of MMA3's K-major B
// operand and z needs no reduction of its own: it is S's column for an all-ones
// value, the reading of z on the same page.
//
// Warp roles: a TMA warp, an MMA warp and sixteen worker warps (four on each TMEM
// lane quarter) that run E1, then E3 together with the feature tiles of the next
// chunk as soon as MMA3 / MMA4 are done, then E2; mbarriers hand over between the
// roles, every wait bounded in time.  E1 touches only the score pieces on or
// below the diagonal.  O has two TMEM buffers (chunk c uses c mod 2), so MMA3 of
// the next chunk need not wait for E2; E2 writes O into a swizzled shared-memory
// tile that one thread stores with TMA.  The pair features are packed bf16
// products, two features of one row per instruction.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "chunk_tc_common.cuh"
#include "trace.h"

namespace la {

namespace {

using namespace tck;

constexpr int kD = 16;                  // width of q and k
constexpr int kDF = 1 + kD + kD * kD;   // 273 features in the page's order
constexpr int kNP = kD * (kD + 1) / 2;  // 136 unordered pairs
constexpr int kDVB = 64;                // value columns per CTA
constexpr int kNV = kDVB + 16;          // O and S_bf16 width: values, normaliser (2), zeros
constexpr int kWarpW = 2;               // first worker warp
constexpr int kThreadsW = 512;          // sixteen worker warps
constexpr int kThreads = 32 * kWarpW + kThreadsW;  // 576
constexpr int kBarW = 1;                // the workers' named barrier
// Feature columns on chip:
//   [0, 136)    pair p = (a, b), a <= b, a-major: x_a x_b, or x_a^2 / sqrt 2 for a = b
//   [136, 152)  x_a
//   152         the constant 1
//   [153, 160)  zero
// and, in the query tile only, the raw q at [160, 176) and the raw k at
// [176, 192) (MMA1's operands; MMA3 never reads them).  16-byte pieces of 8
// columns: pieces 0..16 the pairs, 17..18 x, 19 the constant, 20..23 raw.
constexpr int kFB = 3;                  // 64-column blocks of a feature tile
constexpr int kFCols = 160;             // feature columns the MMAs contract over
// TMEM columns
constexpr uint32_t kColS = 0;           // S^T, 160 columns
constexpr uint32_t kColSc = 160;        // scores (fp32)
constexpr uint32_t kColP = 288;         // P (bf16 pairs), 64 columns
constexpr uint32_t kColO = 352;         // O, two buffers of 80 columns (chunk c uses c mod 2)
constexpr uint32_t kTmemCols = 512;

struct Lay {
    static constexpr uint32_t kRaw = kC * kD * 2;                   // one raw q or k tile
    static constexpr uint32_t kSBBlk = kNV * 128;                   // one 64-column block of S_bf16
    static constexpr uint32_t oPhiQ = 0;                            // query feature tile, 3 x 16 KB
    static constexpr uint32_t oPhiK = oPhiQ + kFB * kBlk;           // key feature tile
    static constexpr uint32_t oSB = oPhiK + kFB * kBlk;             // S_bf16, 3 x 10 KB
    static constexpr uint32_t oV = oSB + kFB * kSBBlk;              // V, two stages
    static constexpr uint32_t oOnes = oV + 2 * kBlk;                // the block after V: ones in column 0
    static constexpr uint32_t oOst = oOnes + kBlk;                  // O staging tile (bf16, swizzled)
    static constexpr uint32_t oQr = oOst + kBlk;                    // raw q, two stages
    static constexpr uint32_t oKr = oQr + 2 * kRaw;                 // raw k, two stages
    static constexpr uint32_t oBar = oKr + 2 * kRaw;
    static constexpr uint32_t oSlot = oBar + 192;                  // TMEM base, abort flag
    static constexpr uint32_t kBytes = oBar + 256;
    static constexpr uint32_t kAlloc = kBytes + 1024;               // + alignment of the base
};
static_assert(Lay::oPhiK % 1024 == 0 && Lay::oSB % 1024 == 0 && Lay::kSBBlk % 1024 == 0 &&
                  Lay::oV % 1024 == 0 && Lay::oOnes % 1024 == 0 && Lay::oOst % 1024 == 0,
              "swizzled blocks need 1024-byte alignment");
static_assert(Lay::kAlloc <= 227 * 1024, "shared memory budget");

enum Bars {
    kFull0 = 0, kFull1 = 1,    // a stage's raw q, k and V landed (TMA)
    kEmpty0 = 2, kEmpty1 = 3,  // a stage read: the workers (raw q, k) and MMA2 / MMA4 (V)
    kPhiReady = 4,             // both feature tiles built
    kSready = 5,               // S_bf16 and the scaled S^T in place (E3, or the initial state)
    kOfree0 = 6,               // E2 has read O buffer 0
    kOfree1 = 7,               // ... and buffer 1
    kPready = 8,               // P in TMEM (E1)
    kScores = 9,               // MMA1 done
    kState = 10,               // MMA1, MMA3, MMA4 done: the feature tiles are free again
    kOut = 11,                 // MMA2 done
    kDrain = 12, kNever = 13, kNumBars = 14
};
static_assert(kNumBars * 8 <= 192, "mbarrier slots");

struct TaylorParams {
    CUtensorMap tmQ, tmK;   // [BH][T][16] bf16, box {16, 128, 1}, no swizzle
    CUtensorMap tmV;        // [BH][T][dv] bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmO;        // O, the same layout (stored from the staging tile)
    __nv_bfloat16* O;       // [BH][T][dv]
    const float* S0;        // [BH][273][dv] in the page's feature order, or null (zero)
    const float* z0;        // [BH][273] or null
    float* S_out;           // final states (same layouts) or null
    float* z_out;
    int H, T, dv, n_dvb;
    int normalize;          // 0 none, 1 divide by the denominator + eps, 2 by max(|.|, 1)
    float eps;
    int* dev_status;
    unsigned long long wait_ns;
    int force_timeout;
    KernelGammas g;
};

// Pair index of (a, b), a <= b, a-major.
__host__ __device__ constexpr int pair_index(int a, int b) { return a * kD - a * (a - 1) / 2 + (b - a); }
static_assert(pair_index(kD - 1, kD - 1) == kNP - 1, "pair count");

// The page rows an on-chip column stands for: (r1, r2) for a pair a < b (the state
// value there is sqrt 2 times the symmetric part of rows r1 = (a, b), r2 = (b, a)),
// (r1, -1) for the rest, (-1, -1) for padding.
__device__ __forceinline__ int2 page_rows(int c) {
    if (c < kNP) {
        int a = 0, p = c;
        while (p >= kD - a) {
            p -= kD - a;
            ++a;
        }
        const int b = a + p;
        return a == b ? make_int2(17 + 17 * a, -1) : make_int2(17 + kD * a + b, 17 + kD * b + a);
    }
    if (c < kNP + kD) return make_int2(1 + c - kNP, -1);
    if (c == kNP + kD) return make_int2(0, -1);
    return make_int2(-1, -1);
}

__device__ __forceinline__ void unpack16(const char* src, float (&x)[kD]) {
    const uint4 u0 = reinterpret_cast<const uint4*>(src)[0];
    const uint4 u1 = reinterpret_cast<const uint4*>(src)[1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

__device__ __forceinline__ void store_piece(char* tile, int r, int piece, const float (&f)[8]) {
    uint4 w;
    w.x = pack_bf16x2(f[0], f[1]);
    w.y = pack_bf16x2(f[2], f[3]);
    w.z = pack_bf16x2(f[4], f[5]);
    w.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(tile + (piece >> 3) * kBlk + sw128_offset(r, (piece & 7) * 8)) = w;
}

// Pieces [P0, P1) of the pair features of one token (row r of a 128-byte-swizzled
// tile): y_a x_b for a < b, y_a x_a / sqrt 2 for a = b, with y = sc x.  Two
// neighbouring features of one row a are one packed bf16 product
// (y_a, y_a) * (x_b, x_b+1): from the input's own bf16 pairs xp when b is even, from
// the pairs shifted by one, xs, when b is odd; the diagonal takes the multiplier
// (y_a / sqrt 2, y_a).  A word that straddles two rows is formed in fp32.  Every
// index is a compile-time constant in the unrolled steps.
template <int P0, int P1>
__device__ __forceinline__ void pair_pieces(char* tile, int r, const float (&y)[kD], const float (&x)[kD],
                                            const __nv_bfloat162 (&yy)[kD], const __nv_bfloat162 (&yd)[kD],
                                            const __nv_bfloat162 (&xp)[kD / 2],
                                            const __nv_bfloat162 (&xs)[kD / 2]) {
    uint32_t word[4];
#pragma unroll
    for (int a = 0; a < kD; ++a)
#pragma unroll
        for (int b = a; b < kD; ++b) {
            const int p = pair_index(a, b);
            if ((p >> 3) < P0 || (p >> 3) >= P1 || (p & 1)) continue;  // words start at even p
            // the second feature of the word: (a, b + 1), or the next row's diagonal
            const bool same_row = b + 1 < kD;
            __nv_bfloat162 w;
            if (same_row) {
                const __nv_bfloat162 m = a == b ? yd[a] : yy[a];
                w = __hmul2(m, (b & 1) ? xs[b >> 1] : xp[b >> 1]);
            } else {
                const float f0 = a == b ? y[a] * x[a] * 0.70710678118654752f : y[a] * x[b];
                const float f1 = y[a + 1] * x[a + 1] * 0.70710678118654752f;
                w = __floats2bfloat162_rn(f0, f1);
            }
            word[(p & 7) >> 1] = *reinterpret_cast<uint32_t*>(&w);
            if ((p & 7) == 6)
                *reinterpret_cast<uint4*>(tile + (p >> 6) * kBlk + sw128_offset(r, ((p >> 3) & 7) * 8)) =
                    make_uint4(word[0], word[1], word[2], word[3]);
        }
}

// Pieces 17..19: y = sc x and the constant sc, zeros after it.
__device__ __forceinline__ void linear_pieces(char* tile, int r, const float (&y)[kD], float sc) {
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = y[e];
    store_piece(tile, r, 17, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = y[8 + e];
    store_piece(tile, r, 18, f);
    *reinterpret_cast<uint4*>(tile + 2 * kBlk + sw128_offset(r, 24)) = make_uint4(pack_bf16x2(sc, 0.f), 0u, 0u, 0u);
}

__global__ void __launch_bounds__(kThreads, 1) chunk_taylor_kernel(const __grid_constant__ TaylorParams p) {
    extern __shared__ __align__(1024) char smem_raw[];
    char* sm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Lay::oSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::oSlot + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x;
    const int bh = unit / p.n_dvb, vb = unit % p.n_dvb, v0 = vb * kDVB;
    const int h = bh % p.H;
    const float l2g = p.g.log2g[h];
    const float gam = p.g.gamma[h];
    const bool unit_gamma = gam == 1.f;
    const int n = (p.T + kC - 1) / kC;
    const uint64_t lim = p.wait_ns;
    constexpr float kRs2 = 0.70710678118654752f;  // 1 / sqrt 2
    constexpr int kPieces = kFCols / 32;          // 32-column pieces of the state

    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&bar[b], 1);
        mbar_init(&bar[kEmpty0], 2);
        mbar_init(&bar[kEmpty1], 2);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&p.tmQ);
        prefetch_tensormap(&p.tmK);
        prefetch_tensormap(&p.tmV);
    }
    if (warp == 1) {
        tmem_alloc(slot, kTmemCols);
        tmem_relinquish();
    }
    // the block after V: a one in column 0 of every token row (MMA2's row sums,
    // MMA4's z row), read through the async proxy; S_bf16 starts at zero (its
    // rows 66..79 stay zero)
    for (int i = tid; i < (int)(kBlk / 16); i += kThreads) {
        const uint32_t one = (i & 7) == ((i >> 3) & 7) ? 0x3F80u : 0u;  // logical piece 0 of row i >> 3
        reinterpret_cast<uint4*>(sm + Lay::oOnes)[i] = make_uint4(one, 0u, 0u, 0u);
    }
    for (int i = tid; i < (int)(kFB * Lay::kSBBlk / 16); i += kThreads)
        reinterpret_cast<uint4*>(sm + Lay::oSB)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t sbase = smem_addr(sm);

    bool forced = false;
    if (p.force_timeout) {  // test hook: a wait on a barrier nothing arrives on
        if (tid == 0 && !mbar_wait(&bar[kNever], 0, lim)) record_status(p.dev_status, LA_ERR_TIMEOUT);
        forced = true;
    }
    int fills[2] = {0, 0};    // producer: TMA fills issued per stage
    bool mma_issued = false;  // issuer: any MMA issued

    if (!forced && n > 0) {
        if (warp == 0 && lane == 0) {
            // ---------------- producer: raw q, k and V of each chunk, two stages
            for (int it = 0; it < n; ++it) {
                const int s = it & 1;
                if (it >= 2 && !mbar_wait_or_abort(&bar[kEmpty0 + s], ((it - 2) >> 1) & 1, lim, abort_flag))
                    break;
                const int y = it * kC;
                mbar_arrive_expect_tx(&bar[kFull0 + s], 2 * Lay::kRaw + kBlk);
                tma_load_3d(sm + Lay::oQr + s * Lay::kRaw, &p.tmQ, 0, y, bh, &bar[kFull0 + s]);
                tma_load_3d(sm + Lay::oKr + s * Lay::kRaw, &p.tmK, 0, y, bh, &bar[kFull0 + s]);
                tma_load_3d(sm + Lay::oV + s * kBlk, &p.tmV, v0, y, bh, &bar[kFull0 + s]);
                ++fills[s];
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer
            const uint64_t dPhiQ = smem_desc_sw128(sbase + Lay::oPhiQ, 16, 1024);        // K-major
            const uint64_t dSB = smem_desc_sw128(sbase + Lay::oSB, 16, 1024);            // K-major
            const uint64_t dPhiK = smem_desc_sw128(sbase + Lay::oPhiK, kBlk, 1024);      // MN-major
            constexpr uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_qs = idesc_bf16(128, kNV, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, kNV, 0, 1);
            constexpr uint32_t id_st = idesc_bf16(128, kFCols, 1, 1);
            for (int it = 0; it < n; ++it) {
                const int s = it & 1;
                // the chunk's feature tiles, the state from E3 of the previous chunk, and
                // this chunk's O buffer read out by E2 two chunks back
                const int ob = it & 1;
                if (!mbar_wait_or_abort(&bar[kPhiReady], it & 1, lim, abort_flag)) break;
                if (!mbar_wait_or_abort(&bar[kSready], it & 1, lim, abort_flag)) break;
                if (it >= 2 && !mbar_wait_or_abort(&bar[kOfree0 + ob], ((it - 2) >> 1) & 1, lim, abort_flag))
                    break;
                fence_after_sync();
                const uint32_t va = sbase + Lay::oV + s * kBlk;
                const uint64_t dVo = smem_desc_sw128(va, sbase + Lay::oOnes - va, 1024);  // MN-major [V | 1]
                // MMA1: scores = q k^T (the raw rows of the query tile)
                mma_ss(tbase + kColSc, desc_adv(dPhiQ, 2 * kBlk + 64), desc_adv(dPhiQ, 2 * kBlk + 96), id_qk, 0u);
                mma_commit(&bar[kScores]);
                mma_issued = true;
                // MMA3: O = phi(Q) S_bf16;  MMA4: S^T += [V | 1]^T phi(K)
#pragma unroll
                for (int kk = 0; kk < kFCols / 16; ++kk)
                    mma_ss(tbase + kColO + ob * kNV, desc_adv(dPhiQ, (kk >> 2) * kBlk + (kk & 3) * 32),
                           desc_adv(dSB, (kk >> 2) * Lay::kSBBlk + (kk & 3) * 32), id_qs, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ss(tbase + kColS, desc_adv(dVo, kk * 2048), desc_adv(dPhiK, kk * 2048), id_st, 1u);
                mma_commit(&bar[kState]);
                // MMA2: O += P [V | 1] once E1 has P in TMEM
                if (!mbar_wait_or_abort(&bar[kPready], it & 1, lim, abort_flag)) break;
                fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ts(tbase + kColO + ob * kNV, tbase + kColP + kk * 8, desc_adv(dVo, kk * 2048), id_pv, 1u);
                mma_commit(&bar[kOut]);
                mma_commit(&bar[kEmpty0 + s]);
            }
        } else if (warp >= kWarpW) {
            // ---------------- workers: four warps on each TMEM lane quarter
            const int t = tid - 32 * kWarpW;          // 0 .. 511
            const int q4 = warp & 3;                  // TMEM lane quarter of this warp
            const int sub = t >> 7;                   // which of the quarter's four warps (warp-uniform)
            const int row = q4 * 32 + lane;           // TMEM lane of this thread
            const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
            // this warp's 32-column pieces of the state: sub and sub + 4
            const int n_own = sub + 4 < kPieces ? 2 : 1;

            // S^T <- the initial state in the kernel's coordinates (lanes 0..63: value
            // columns v0 + lane, lane 64: z; a pair column takes the two page rows'
            // sum over sqrt 2; other lanes zero)
            {
                const float* src = nullptr;
                size_t stride = 0;
                if (row < kDVB && p.S0) {
                    src = p.S0 + (size_t)bh * kDF * p.dv + v0 + row;
                    stride = p.dv;
                } else if (row == kDVB && p.z0) {
                    src = p.z0 + (size_t)bh * kDF;
                    stride = 1;
                }
                for (int k = 0; k < n_own; ++k) {
                    const int c0 = (sub + 4 * k) * 32;
                    uint32_t r[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int2 pr = page_rows(c0 + e);
                        float x = 0.f;
                        if (src && pr.x >= 0) {
                            x = src[pr.x * stride];
                            if (pr.y >= 0) x = (x + src[pr.y * stride]) * kRs2;
                        }
                        r[e] = __float_as_uint(x);
                    }
                    tmem_st32(tbase + lane_off + kColS + c0, r);
                }
                tmem_st_wait();
                fence_before_sync();
                named_bar_sync(kBarW, kThreadsW);
                fence_after_sync();
            }

            // E3: S^T -> the bf16 B operand of MMA3 (K-major: row n = value column n;
            // rows 64 and 65 = z's bf16 value and its residual), then S^T *= decay
            // (skipped when `scale` is false).  Lanes 65..127 hold nothing.
            auto e3 = [&](float decay, bool scale) {
                if (q4 == 3) return;  // warp-uniform
                for (int hp = sub; hp < 2 * kPieces; hp += 4) {  // 16-column halves: three or two a warp
                    const int c0 = hp * 16;
                    uint32_t r[16];
                    tmem_ld16(tbase + lane_off + kColS + c0, r);
                    tmem_ld_wait();
                    char* base = sm + Lay::oSB + (c0 >> 6) * Lay::kSBBlk;
                    const int cb = c0 & 63;
                    if (row < kDVB) {
#pragma unroll
                        for (int e8 = 0; e8 < 16; e8 += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(r[e8 + 0]), __uint_as_float(r[e8 + 1]));
                            w.y = pack_bf16x2(__uint_as_float(r[e8 + 2]), __uint_as_float(r[e8 + 3]));
                            w.z = pack_bf16x2(__uint_as_float(r[e8 + 4]), __uint_as_float(r[e8 + 5]));
                            w.w = pack_bf16x2(__uint_as_float(r[e8 + 6]), __uint_as_float(r[e8 + 7]));
                            *reinterpret_cast<uint4*>(base + sw128_offset(row, cb + e8)) = w;
                        }
                    } else if (row == kDVB) {
#pragma unroll
                        for (int e8 = 0; e8 < 16; e8 += 8) {
                            uint32_t hw[4], lw[4];
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float x0 = __uint_as_float(r[e8 + e]), x1 = __uint_as_float(r[e8 + e + 1]);
                                const uint32_t hi = pack_bf16x2(x0, x1);  // x0 in the low half
                                hw[e >> 1] = hi;
                                lw[e >> 1] = pack_bf16x2(x0 - __uint_as_float(hi << 16),
                                                         x1 - __uint_as_float(hi & 0xFFFF0000u));
                            }
                            *reinterpret_cast<uint4*>(base + sw128_offset(kDVB, cb + e8)) =
                                make_uint4(hw[0], hw[1], hw[2], hw[3]);
                            *reinterpret_cast<uint4*>(base + sw128_offset(kDVB + 1, cb + e8)) =
                                make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        }
                    }
                    if (scale) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * decay);
                        tmem_st16(tbase + lane_off + kColS + c0, r);
                    }
                }
                if (scale) tmem_st_wait();
            };

            // The feature tiles of chunk `it` (stage s): queries xi-scaled (with the raw q
            // and k for MMA1), keys zeta-scaled; rows past the end are zero.  Worker t
            // builds row t mod 128: sub 0 / 1 the queries' pair pieces 0..10 / the rest
            // with x, the constant and the raw rows; sub 2 / 3 the same of the keys.
            auto build_phi = [&](int s, int L) {
                const int r = t & (kC - 1);
                const bool is_q = sub < 2;
                const char* src = sm + (is_q ? Lay::oQr : Lay::oKr) + s * Lay::kRaw + r * (kD * 2);
                char* tile = sm + (is_q ? Lay::oPhiQ : Lay::oPhiK);
                float sc = 0.f;  // xi_r or zeta_r, zero past the end
                if (r < L) sc = unit_gamma ? 1.f : gamma_pow(l2g, (float)(is_q ? r + 1 : L - 1 - r));
                float x[kD], y[kD];
                unpack16(src, x);
                __nv_bfloat162 xp[kD / 2], xs[kD / 2], yy[kD], yd[kD];
#pragma unroll
                for (int e = 0; e < kD / 2; ++e) {
                    xp[e] = reinterpret_cast<const __nv_bfloat162*>(src)[e];  // (x_2e, x_2e+1)
                    xs[e] = __floats2bfloat162_rn(x[2 * e + 1], 2 * e + 2 < kD ? x[2 * e + 2] : 0.f);
                }
#pragma unroll
                for (int a = 0; a < kD; ++a) {
                    y[a] = x[a] * sc;
                    yy[a] = __float2bfloat162_rn(y[a]);
                    yd[a] = __floats2bfloat162_rn(y[a] * 0.70710678118654752f, y[a]);
                }
                if ((sub & 1) == 0) {
                    pair_pieces<0, 11>(tile, r, y, x, yy, yd, xp, xs);
                } else {
                    pair_pieces<11, 17>(tile, r, y, x, yy, yd, xp, xs);
                    linear_pieces(tile, r, y, sc);
                    if (is_q) {  // the raw rows (the tile loads zero past the end of the sequence)
                        const uint4* qr = reinterpret_cast<const uint4*>(src);
                        const uint4* kr = reinterpret_cast<const uint4*>(sm + Lay::oKr + s * Lay::kRaw + r * (kD * 2));
                        *reinterpret_cast<uint4*>(tile + 2 * kBlk + sw128_offset(r, 32)) = qr[0];
                        *reinterpret_cast<uint4*>(tile + 2 * kBlk + sw128_offset(r, 40)) = qr[1];
                        *reinterpret_cast<uint4*>(tile + 2 * kBlk + sw128_offset(r, 48)) = kr[0];
                        *reinterpret_cast<uint4*>(tile + 2 * kBlk + sw128_offset(r, 56)) = kr[1];
                    }
                }
            };

            // E1 on score piece sub (columns j = 32 sub ..) of query row i: the Taylor
            // kernel times gamma^(i - j) for j <= i < L, else 0, as 16 bf16 pairs in P.
            // A warp's 32 rows and a piece's 32 columns are one 32 x 32 block for every
            // lane: above the diagonal the piece is zero (no load), below it no column
            // needs the mask.
            auto e1 = [&](int L) {
                const int cc = 32 * sub;
                const int i = row;
                uint32_t out[16];
                if (sub > q4) {  // warp-uniform: above the diagonal
#pragma unroll
                    for (int e = 0; e < 16; ++e) out[e] = 0u;
                } else if (sub < q4 && L == kC && unit_gamma) {  // below the diagonal, no mask, no decay
#pragma unroll
                    for (int h16 = 0; h16 < 32; h16 += 16) {
                        uint32_t r[16];
                        tmem_ld16(tbase + lane_off + kColSc + cc + h16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float s0 = __uint_as_float(r[e]), s1 = __uint_as_float(r[e + 1]);
                            out[(h16 + e) >> 1] = pack_bf16x2(fmaf(s0, fmaf(0.5f, s0, 1.f), 1.f),
                                                              fmaf(s1, fmaf(0.5f, s1, 1.f), 1.f));
                        }
                    }
                } else {
                    const bool diag = sub == q4;
                    const bool live = i < L;
                    const int jt = min(i, cc + 31);
                    float w = unit_gamma ? 1.f : gamma_pow(l2g, (float)(i - jt));
#pragma unroll
                    for (int h16 = 16; h16 >= 0; h16 -= 16) {  // the upper 16 columns first (the decay runs down)
                        uint32_t r[16];
                        tmem_ld16(tbase + lane_off + kColSc + cc + h16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 14; e >= 0; e -= 2) {  // each pair packed at once
                            const int j = cc + h16 + e;
                            const float s1 = __uint_as_float(r[e + 1]), s0 = __uint_as_float(r[e]);
                            float v1 = fmaf(s1, fmaf(0.5f, s1, 1.f), 1.f);
                            float v0 = fmaf(s0, fmaf(0.5f, s0, 1.f), 1.f);
                            const bool in1 = live && (!diag || j + 1 <= i), in0 = live && (!diag || j <= i);
                            if (!unit_gamma) {
                                v1 *= w;
                                if (in1) w *= gam;
                                v0 *= w;
                                if (in0) w *= gam;
                            }
                            out[(h16 + e) >> 1] = pack_bf16x2(in0 ? v0 : 0.f, in1 ? v1 : 0.f);
                        }
                    }
                }
                tmem_st16(tbase + lane_off + kColP + (cc >> 1), out);
                tmem_st_wait();
            };

            // E2: O rows, divided by the normaliser, into the staging tile (16 value
            // columns a warp); one thread then stores the tile with TMA
            auto e2 = [&](int it) {
                const uint32_t ocol = tbase + lane_off + kColO + (it & 1) * kNV;
                uint32_t r[16];
                tmem_ld16(ocol + 16 * sub, r);
                float inv = 1.f;
                if (p.normalize) {
                    const float den = __uint_as_float(tmem_ld1(ocol + kDVB)) +
                                      __uint_as_float(tmem_ld1(ocol + kDVB + 1));
                    tmem_ld_wait();
                    inv = 1.f / norm_den(den, p.normalize, p.eps);
                } else {
                    tmem_ld_wait();
                }
                char* ost = sm + Lay::oOst;
#pragma unroll
                for (int e8 = 0; e8 < 16; e8 += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(r[e8 + 0]) * inv, __uint_as_float(r[e8 + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(r[e8 + 2]) * inv, __uint_as_float(r[e8 + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(r[e8 + 4]) * inv, __uint_as_float(r[e8 + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(r[e8 + 6]) * inv, __uint_as_float(r[e8 + 7]) * inv);
                    *reinterpret_cast<uint4*>(ost + sw128_offset(row, 16 * sub + e8)) = w;
                }
            };

            // The final state in the page's feature order (z from the first value block
            // only): a pair column gives rows (a, b) and (b, a) its value over sqrt 2,
            // plus the decayed antisymmetric part of the initial state.
            auto write_exit_state = [&]() {
                if (q4 == 3 || (!p.S_out && !p.z_out)) return;  // warp-uniform
                float* dst = nullptr;
                const float* src0 = nullptr;
                size_t stride = 0;
                if (row < kDVB && p.S_out) {
                    dst = p.S_out + (size_t)bh * kDF * p.dv + v0 + row;
                    src0 = p.S0 ? p.S0 + (size_t)bh * kDF * p.dv + v0 + row : nullptr;
                    stride = p.dv;
                } else if (row == kDVB && vb == 0 && p.z_out) {
                    dst = p.z_out + (size_t)bh * kDF;
                    src0 = p.z0 ? p.z0 + (size_t)bh * kDF : nullptr;
                    stride = 1;
                }
                const float gT = unit_gamma ? 1.f : gamma_pow(l2g, (float)p.T);
                for (int k = 0; k < n_own; ++k) {
                    const int c0 = (sub + 4 * k) * 32;
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + kColS + c0, r);
                    tmem_ld_wait();
                    if (!dst) continue;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int2 pr = page_rows(c0 + e);
                        if (pr.x < 0) continue;
                        const float x = __uint_as_float(r[e]);
                        if (pr.y < 0) {
                            dst[pr.x * stride] = x;
                        } else {
                            const float anti = src0 ? 0.5f * gT * (src0[pr.x * stride] - src0[pr.y * stride]) : 0.f;
                            dst[pr.x * stride] = x * kRs2 + anti;
                            dst[pr.y * stride] = x * kRs2 - anti;
                        }
                    }
                }
            };

            // E3 for chunk `it` (or the initial state, it = -1) and the feature tiles
            // of chunk it + 1, then hand both over to the MMA warp
            auto state_and_features = [&](int it) -> bool {
                const int nx = it + 1;
                const int Ln = min(kC, p.T - nx * kC);
                e3(unit_gamma ? 1.f : gamma_pow(l2g, (float)Ln), !unit_gamma);
                const int s = nx & 1;
                const bool ok = mbar_wait_or_abort(&bar[kFull0 + s], (nx >> 1) & 1, lim, abort_flag);
                if (named_bar_or(kBarW, kThreadsW, !ok)) return false;
                build_phi(s, Ln);
                fence_proxy_async_smem();
                fence_before_sync();
                named_bar_sync(kBarW, kThreadsW);
                if (t == 0) {
                    mbar_arrive(&bar[kSready]);
                    mbar_arrive(&bar[kPhiReady]);
                    mbar_arrive(&bar[kEmpty0 + s]);  // the stage's raw rows are read
                }
                return true;
            };

            // it = -1 hands over the initial state and the first chunk's features
            for (int it = -1; it < n; ++it) {
                const int L = it >= 0 ? min(kC, p.T - it * kC) : 0;
                (void)L;
                bool ok = true;
                if (it >= 0) {
                    // ---- E1 once MMA1 is done (MMA3 / MMA4 run beside it)
                    ok = mbar_wait_or_abort(&bar[kScores], it & 1, lim, abort_flag);
                    if (named_bar_or(kBarW, kThreadsW, !ok)) break;
                    fence_after_sync();
                    e1(L);
                    fence_before_sync();
                    named_bar_sync(kBarW, kThreadsW);
                    if (t == 0) mbar_arrive(&bar[kPready]);
                    // ---- once MMA3 and MMA4 are done (MMA2 runs beside it)
                    ok = mbar_wait_or_abort(&bar[kState], it & 1, lim, abort_flag);
                    if (named_bar_or(kBarW, kThreadsW, !ok)) break;
                    fence_after_sync();
                }
                // ---- E3 and the next chunk's feature tiles, or the final state
                if (it + 1 < n) {
                    if (!state_and_features(it)) break;
                } else {
                    write_exit_state();
                }
                if (it >= 0) {
                    // ---- E2 once MMA2 is done (and the previous chunk's store has read the
                    // staging tile); then the O buffer is free for chunk it + 2
                    if (t == 0) bulk_wait_read0();
                    ok = mbar_wait_or_abort(&bar[kOut], it & 1, lim, abort_flag);
                    if (named_bar_or(kBarW, kThreadsW, !ok)) break;
                    fence_after_sync();
                    e2(it);
                    fence_proxy_async_smem();
                    fence_before_sync();
                    named_bar_sync(kBarW, kThreadsW);
                    if (t == 0) {
                        mbar_arrive(&bar[kOfree0 + (it & 1)]);
                        tma_store_3d(&p.tmO, v0, it * kC, bh, sm + Lay::oOst);  // rows past T are not written
                        bulk_commit();
                    }
                }
            }
            if (t == 0) bulk_wait0();  // the last stores are done before the CTA leaves
        }
    }

    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (*abort_flag || forced) {
        record_status(p.dev_status, LA_ERR_TIMEOUT);
        if (warp == 0 && lane == 0) {  // our own TMA fills must land before the smem is released
            for (int s = 0; s < 2; ++s)
                if (fills[s] > 0) mbar_wait(&bar[kFull0 + s], (fills[s] - 1) & 1, lim);
        }
        if (warp == 1 && lane == 0 && mma_issued) {  // and our MMAs before TMEM is freed
            mma_commit(&bar[kDrain]);
            mbar_wait(&bar[kDrain], 0, lim);
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

bool taylor_supported(const ChunkArgs& a) {
    return a.taylor && a.bf16 && a.dk == kD && a.dv > 0 && a.dv % kDVB == 0 && !a.noncausal &&
           !a.phi && !a.log_a && (a.chunk == 0 || a.chunk == kC) && tck::tc_arch_ok();
}

int taylor_feature_dim(int d) { return 1 + d + d * d; }

cudaError_t launch_chunk_taylor(const ChunkArgs& a, const KernelGammas& g, cudaStream_t s) {
    if (!taylor_supported(a)) return cudaErrorInvalidValue;
    TaylorParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int BH = a.B * a.H;
    if (!tck::make_map_box(&prm.tmQ, a.Q, BH, a.T, kD, kD, false) ||
        !tck::make_map_box(&prm.tmK, a.K, BH, a.T, kD, kD, false) ||
        !tck::make_map(&prm.tmV, a.V, BH, a.T, a.dv) || !tck::make_map(&prm.tmO, a.O, BH, a.T, a.dv))
        return cudaErrorInvalidValue;
    prm.O = static_cast<__nv_bfloat16*>(a.O);
    prm.S0 = a.S0;
    prm.z0 = a.z0;
    prm.S_out = a.S_out;
    prm.z_out = a.z_out;
    prm.H = a.H;
    prm.T = a.T;
    prm.dv = a.dv;
    prm.n_dvb = a.dv / kDVB;
    prm.normalize = norm_mode(a.normalize, a.floor_norm);
    prm.eps = a.eps;
    prm.dev_status = a.dev_status;
    prm.wait_ns = 2000000000ull;
    if (opt_force_timeout()) {
        prm.force_timeout = 1;
        prm.wait_ns = 1000000ull;  // 1 ms
    }
    prm.g = g;
    cudaError_t e = cudaFuncSetAttribute(chunk_taylor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::kAlloc);
    if (e != cudaSuccess) return e;
    TraceScope trace("chunk_taylor_kernel", s);
    chunk_taylor_kernel<<<BH * prm.n_dvb, kThreads, Lay::kAlloc, s>>>(prm);
    return cudaGetLastError();
}

}  // namespace la
