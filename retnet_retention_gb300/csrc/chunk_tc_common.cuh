// Definitions shared by the tensor-core chunk kernels (chunk_tc.cu: the
// lockstep kernel; chunk_tc_ws.cu: the warp-specialised pipeline).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace la {
namespace tck {

using namespace tc;

constexpr int kC = 128;           // chunk length (= MMA M)
constexpr uint32_t kColP = 0;     // scores (fp32, 128 cols) then P (bf16 pairs, 64 cols)
constexpr uint32_t kBlk = 16384;  // one [128 rows x 64 bf16] swizzled block
constexpr int kFoldMax = 4;      // most segments per sequence whose entry states the output walk folds

enum Mode { kFull = 0, kStateOnly = 1, kNonCausal = 2 };

struct TcParams {
    CUtensorMap tmQ, tmK, tmV;  // [BH][T][d] bf16, box {64, 128, 1}, 128B swizzle
    __nv_bfloat16* O;           // [BH][T][dv]
    const float* S_in;          // entry states or nullptr (zero)
    const float* z_in;
    float* S_out;               // final states or nullptr
    float* z_out;
    int in_nseg;                // entry-state index = bh * in_nseg + seg
    int out_nseg;               // exit-state index = bh * out_nseg + (out_last_only ? 0 : seg)
    int out_last_only;
    int H, T, dv;
    int n_dvb;                  // value-column blocks per sequence
    int seg_chunks;             // chunks per segment
    int n_seg;                  // segments per sequence
    int mode;
    int normalize;              // 0 none, 1 divide by q^.z + eps, 2 by max(|q^.z|, 1)
    int track_z;                // carry the normaliser state z (normalising, or z_out wanted)
    int phi;
    float eps;
    // in_agg: S_in / z_in hold the segments' own contributions (state walk), and the
    // output walk folds them into its entry state itself, starting from S0 / z0
    // (null = zero): entry_q = gamma^len entry_{q-1} + agg_{q-1}, len = seg_chunks * C
    int in_agg;
    const float* S0;
    const float* z0;
    // per-token decay (null: the per-head gammas): per chunk of every sequence,
    // 128 cumulative log2 decays then 128 decays ([BH][n_chunks][2][128] fp32,
    // written by gate_prep_kernel), and each segment's total log2 decay
    // ([BH][n_seg]: written by the state walk, read by the fold and the scan)
    const float* gate;
    float* seg_l2;
    int* dev_status;
    unsigned long long wait_ns;
    int force_timeout;
    // every head's gamma < 1 with gamma^(C-1) >= 2^-64, no feature map, no normaliser,
    // z not carried: the pipelined kernel's factored-decay build
    int fact;
    // reversed time (factored-decay build only): the sums run over s >= t, the
    // chunks are walked from the end of the sequence (chunk c covers rows
    // T - (c + 1) C .. T - c C - 1, the last one starting before row 0, where the
    // tiles read zeros), and tile row r stands at position C - 1 - r of its chunk
    // in the reversed sequence.  The initial state enters at the end, and the
    // final state is the one after row 0.
    int rev;
    // per-token decay, output walk: [BH][n_chunks] flags from gate_prep_kernel (1: the
    // chunk's decay leaves the factored build's range), read by the pick kernel
    const int* gate_flags;
    int o_align32;  // O's base is 32-byte aligned (rows and column blocks then are too)
    KernelGammas g;
};

// A compile-time bool for generic lambdas (one instantiation per value).
template <bool B>
struct BoolC {
    static constexpr bool value = B;
};

__device__ __forceinline__ void record_status(int* st, int code) {
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float phi_f(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// phi = elu + 1 on a bf16 pair: relu(x) + e^min(x, 0), i.e. x + 1 above zero
// (rounded once, in bf16) and e^x at or below it (e^x in fp32, then rounded).
__device__ __forceinline__ __nv_bfloat162 phi_bf16x2(__nv_bfloat162 x) {
    const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
    const float2 m = __bfloat1622float2(__hmin2(x, zero));
    return __hadd2(__hmax2(x, zero), __floats2bfloat162_rn(__expf(m.x), __expf(m.y)));
}

// phi on rows < L of a [128 x 64*nblk] K-major swizzled tile, rows >= L set
// to zero (phi(0) = 1, so rows past the end of the sequence must be cleared),
// by `nthr` threads (this one is `t`).
__device__ __forceinline__ void phi_rows(char* tile, int nblk, int L, int t, int nthr) {
    const int n16 = nblk * (kBlk / 16);
    for (int idx = t; idx < n16; idx += nthr) {
        const int r = (idx >> 3) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile) + idx;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < L) {
            u = *p;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = phi_bf16x2(h[e]);
        }
        *p = u;
    }
}

// The same over NT tiles of NBLK blocks each by exactly NTHR threads (a
// multiple of 128 that divides a block's 1024 pieces), with every load issued
// before the first exp and every store after the last, so one thread has all
// its pieces in flight at once.
template <int NT, int NBLK, int NTHR>
__device__ __forceinline__ void phi_rows_all(char* const (&tiles)[NT], int L, int t) {
    static_assert(NTHR % 128 == 0 && (kBlk / 16) % NTHR == 0, "thread count");
    constexpr int kPer = NBLK * (kBlk / 16) / NTHR;  // 16-byte pieces per thread and tile
    uint4 u[NT][kPer];
#pragma unroll
    for (int q = 0; q < NT; ++q)
#pragma unroll
        for (int k = 0; k < kPer; ++k) u[q][k] = reinterpret_cast<const uint4*>(tiles[q])[t + NTHR * k];
#pragma unroll
    for (int q = 0; q < NT; ++q)
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int r = ((t + NTHR * k) >> 3) & 127;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u[q][k]);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = phi_bf16x2(h[e]);
            if (r >= L) u[q][k] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
    for (int q = 0; q < NT; ++q)
#pragma unroll
        for (int k = 0; k < kPer; ++k) reinterpret_cast<uint4*>(tiles[q])[t + NTHR * k] = u[q][k];
}

// Row r of a [128 x 64*NBLK] K-major swizzled tile times fac(r), by exactly
// NTHR threads, every load issued before the first multiply.
template <int NBLK, int NTHR, typename F>
__device__ __forceinline__ void scale_rows_all(char* tile, F fac, int t) {
    static_assert(NTHR % 128 == 0 && (kBlk / 16) % NTHR == 0, "thread count");
    constexpr int kPer = NBLK * (kBlk / 16) / NTHR;
    uint4 u[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) u[k] = reinterpret_cast<const uint4*>(tile)[t + NTHR * k];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const float f = fac(((t + NTHR * k) >> 3) & 127);
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u[k]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(h[e]);
            h[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
        }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) reinterpret_cast<uint4*>(tile)[t + NTHR * k] = u[k];
}

// Q^ = xi . Q in place over a [128 x DK] K-major swizzled bf16 tile by 128
// threads, and per row out[r] = xi_r (q_r . z) in fp32 from the tile before it
// is rounded: the inter-chunk part of the normaliser without the bf16 rounding
// of xi_r q_r (with signed features q . z can be a small difference of large
// terms).  Thread t holds 16-byte piece t & 7 of rows (t >> 3) + 16 m, m < 8,
// in every 64-column block; the 8 pieces of a row sit in 8 consecutive lanes.
template <int DK, typename F>
__device__ __forceinline__ void scale_rows_dot(char* tile, F fac, const float* z, float* out, int t) {
    const int pc = t & 7;
#pragma unroll 1
    for (int m = 0; m < 8; ++m) {
        const int r = (t >> 3) + 16 * m;
        const int lc = pc ^ (r & 7);  // logical 8-column group of the physical piece
        const float f = fac(r);
        float acc = 0.f;
#pragma unroll
        for (int b = 0; b < DK / 64; ++b) {
            uint4* p = reinterpret_cast<uint4*>(tile + b * kBlk) + (r * 8 + pc);
            uint4 u = *p;
            const float4 za = *reinterpret_cast<const float4*>(z + b * 64 + lc * 8);
            const float4 zb = *reinterpret_cast<const float4*>(z + b * 64 + lc * 8 + 4);
            __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
            const float2 x0 = __bfloat1622float2(hv[0]), x1 = __bfloat1622float2(hv[1]);
            const float2 x2 = __bfloat1622float2(hv[2]), x3 = __bfloat1622float2(hv[3]);
            acc = fmaf(x0.x, za.x, acc); acc = fmaf(x0.y, za.y, acc);
            acc = fmaf(x1.x, za.z, acc); acc = fmaf(x1.y, za.w, acc);
            acc = fmaf(x2.x, zb.x, acc); acc = fmaf(x2.y, zb.y, acc);
            acc = fmaf(x3.x, zb.z, acc); acc = fmaf(x3.y, zb.w, acc);
            hv[0] = __floats2bfloat162_rn(x0.x * f, x0.y * f);
            hv[1] = __floats2bfloat162_rn(x1.x * f, x1.y * f);
            hv[2] = __floats2bfloat162_rn(x2.x * f, x2.y * f);
            hv[3] = __floats2bfloat162_rn(x3.x * f, x3.y * f);
            *p = u;
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (pc == 0) out[r] = f * acc;
    }
}

// K^ = zeta . K in place over a [128 x DK] K-major swizzled bf16 tile by 128
// threads (row r times fac(r) = zeta_r, 0 for rows >= L), and the fp32 column sums
// of zeta_r k_r taken from the unscaled values (the normaliser state's update,
// without the bf16 rounding of zeta_r k_r).  Each 64-column block has its own
// NT = 128 / (DK / 64) threads; thread t' of a block holds 16-byte piece t' & 7
// of rows (t' >> 3) + (NT / 8) m, so it always holds the same logical 8-column
// group lc = (t' & 7) ^ ((t' >> 3) & 7), and the four lanes of a warp with the
// same group (lanes l, l ^ 9, l ^ 18, l ^ 27) add their sums.  Lanes 0-7 of
// each warp then store the warp's sums into part ([256/DK][DK] floats, slot =
// the warp's index within its block: the layout colsum_total() reads); the
// caller synchronises the 128 threads before reading them.
template <int DK, typename F>
__device__ __forceinline__ void scale_rows_zsum(char* tile, F fac, float* part, int t) {
    constexpr int NT = 128 / (DK / 64);  // threads per block
    constexpr int NP = 1024 / NT;        // pieces per thread
    const int b = t / NT, tb = t % NT;
    const int pc = tb & 7, rg = tb >> 3;
    uint4* base = reinterpret_cast<uint4*>(tile + b * kBlk) + rg * 8 + pc;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 2
    for (int m = 0; m < NP; ++m) {
        const int r = rg + (NT / 8) * m;
        const float f = fac(r);
        uint4 u = base[m * NT];  // NT / 8 rows of 8 pieces further on
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(hv[e]);
            const float px = x.x * f, py = x.y * f;
            acc[2 * e] += px;
            acc[2 * e + 1] += py;
            hv[e] = __floats2bfloat162_rn(px, py);
        }
        base[m * NT] = u;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 9);
        acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 18);
    }
    const int l = t & 31;
    if (l < 8) {
        const int lc = l ^ (rg & 7);  // lane l < 8: piece l of row group rg
        float4* dst = reinterpret_cast<float4*>(part + (tb >> 5) * DK + b * 64 + lc * 8);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// A factor f as a pair of bf16x2 words (both halves equal): h = bf16(f) and
// l = bf16(f - h), for scale_rows_hl.
__device__ __forceinline__ void split_bf16x2(float f, uint32_t& h, uint32_t& l) {
    const __nv_bfloat16 fh = __float2bfloat16_rn(f);
    const __nv_bfloat16 fl = __float2bfloat16_rn(f - __bfloat162float(fh));
    const uint32_t uh = __bfloat16_as_ushort(fh), ul = __bfloat16_as_ushort(fl);
    h = uh | (uh << 16);
    l = ul | (ul << 16);
}

// Row r of a [128 x 64*NBLK] K-major swizzled bf16 tile times its factor, in
// place, by exactly NTHR threads, in packed bf16 arithmetic: each element x
// becomes fma(x, h, bf16(x l)) with the factor split as h + l (split_bf16x2),
// one rounding of a sum within about 2^-17 (relative) of x f: the fp32 product
// rounded to bf16 but for near-ties, at eight instructions per 16-byte piece
// instead of about twenty.  Thread t holds piece t & 7 of rows
// (t >> 3) + (NTHR / 8) m, m < 1024 / NTHR, of every block (a row is one
// 128-byte line, so the swizzle keeps pieces in their row); h[m], l[m] are that
// row's factor.  Eight pieces are loaded before any is computed.
template <int NBLK, int NTHR>
__device__ __forceinline__ void scale_rows_hl(char* tile, const uint32_t (&h)[1024 / NTHR],
                                              const uint32_t (&l)[1024 / NTHR], int t) {
    static_assert(NTHR % 8 == 0 && 1024 % NTHR == 0, "thread count");
    constexpr int R = 1024 / NTHR;
    constexpr int kB = R < 8 ? R : 8;
    uint4* base = reinterpret_cast<uint4*>(tile) + t;
#pragma unroll
    for (int b = 0; b < NBLK; ++b)
#pragma unroll
        for (int m0 = 0; m0 < R; m0 += kB) {
            uint4 u[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j) u[j] = base[b * 1024 + (m0 + j) * NTHR];
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                uint32_t* x = reinterpret_cast<uint32_t*>(&u[j]);
                const __nv_bfloat162 hh = *reinterpret_cast<const __nv_bfloat162*>(&h[m0 + j]);
                const __nv_bfloat162 ll = *reinterpret_cast<const __nv_bfloat162*>(&l[m0 + j]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&x[e]);
                    const __nv_bfloat162 y = __hfma2(v, hh, __hmul2(v, ll));
                    x[e] = *reinterpret_cast<const uint32_t*>(&y);
                }
            }
#pragma unroll
            for (int j = 0; j < kB; ++j) base[b * 1024 + (m0 + j) * NTHR] = u[j];
        }
}

// In-place pass over a [128 x 64*nblk] K-major swizzled tile by `nthr`
// threads (this one is `t`): apply phi (optional) and multiply row r by
// fac(r).  Rows are whole 128-byte lines, so the swizzle never moves an
// element to another row.
template <typename F>
__device__ __forceinline__ void row_pass(char* tile, int nblk, bool apply_phi, F fac, int t,
                                         int nthr) {
    const int n16 = nblk * (kBlk / 16);
    for (int idx = t; idx < n16; idx += nthr) {
        const int r = (idx >> 3) & 127;
        uint4* p = reinterpret_cast<uint4*>(tile) + idx;
        uint4 u = *p;
        const float f = fac(r);
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
        if (apply_phi) {
            const __nv_bfloat162 ff = __float2bfloat162_rn(f);  // f is 0 or 1 here
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __hmul2(phi_bf16x2(h[e]), ff);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __bfloat1622float2(h[e]);
                h[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
            }
        }
        *p = u;
    }
}

// Column sums of a [128 x DK] K-major swizzled bf16 tile (over its rows) by 128
// threads: thread t sums column pair (2 cp, 2 cp + 1), cp = t mod DK/2, over one
// of 256/DK row groups; a warp reads whole 128-byte rows (conflict-free).
// Partials go to `part` ([256/DK][DK] floats); the caller synchronises the 128
// threads and then reads colsum_total().
// Each row j < L is weighted by zeta_j = gamma^(L-1-j) in fp32 (rows >= L get
// weight 0), on the tile before it is scaled: sum_j zeta_j k^_j without the
// bf16 rounding of zeta_j k^_j, which signed features would otherwise turn into
// a large error of q^ . z after cancellation.  The weights are a running
// product from the group's last row upwards (zeta grows by 1/gamma per row
// towards the top, so the product runs downwards in gamma and never overflows).
template <int DK>
__device__ __forceinline__ void colsum_partial_decayed(const char* tile, int t, float* part, int L,
                                                       float l2g, float gam) {
    constexpr int kPairs = DK / 2;
    constexpr int kGroups = 128 / kPairs;
    constexpr int kRows = 128 / kGroups;
    const int cp = t % kPairs, grp = t / kPairs;
    const int col = 2 * cp;
    const char* base = tile + (col >> 6) * kBlk;
    const int jtop = grp * kRows + kRows - 1;
    float w = gamma_pow(l2g, (float)max(L - 1 - jtop, 0));
    float ax = 0.f, ay = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < kRows; ++jj) {
        const int j = jtop - jj;
        const float2 f = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(base + sw128_offset(j, col & 63)));
        const bool in = j < L;
        const float wj = in ? w : 0.f;
        ax = fmaf(wj, f.x, ax);
        ay = fmaf(wj, f.y, ay);
        w = in ? w * gam : w;
    }
    part[grp * DK + col] = ax;
    part[grp * DK + col + 1] = ay;
}
// The same with gamma = 1: plain column sums over all 128 rows (rows past the
// end of the sequence hold zeros: the copy's fill, or phi's clearing).
template <int DK>
__device__ __forceinline__ void colsum_partial(const char* tile, int t, float* part) {
    constexpr int kPairs = DK / 2;
    constexpr int kGroups = 128 / kPairs;
    constexpr int kRows = 128 / kGroups;
    const int cp = t % kPairs, grp = t / kPairs;
    const int col = 2 * cp;
    const char* base = tile + (col >> 6) * kBlk;
    float ax = 0.f, ay = 0.f;
#pragma unroll 8
    for (int j = grp * kRows; j < (grp + 1) * kRows; ++j) {
        const float2 f = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(base + sw128_offset(j, col & 63)));
        ax += f.x;
        ay += f.y;
    }
    part[grp * DK + col] = ax;
    part[grp * DK + col + 1] = ay;
}
template <int DK>
__device__ __forceinline__ float colsum_total(const float* part, int d) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < 128 / (DK / 2); ++g) s += part[g * DK + d];
    return s;
}

// Host: 3-D TMA map [BH][T][d] bf16, box {64, 128, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int BH, int T, int d);
// [BH][T][d] bf16 with a box of box_x x 128 rows, 128-byte swizzle or none.
bool make_map_box(CUtensorMap* m, const void* base, int BH, int T, int d, int box_x, bool swizzle);
// The tensor-map encoder is reachable and the device is sm_103.
bool tc_arch_ok();

}  // namespace tck
}  // namespace la
