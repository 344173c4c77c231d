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
    int normalize;
    int track_z;                // carry the normaliser state z (normalising, or z_out wanted)
    int phi;
    float eps;
    // in_agg: S_in / z_in hold the segments' own contributions (state walk), and the
    // output walk folds them into its entry state itself, starting from S0 / z0
    // (null = zero): entry_q = gamma^len entry_{q-1} + agg_{q-1}, len = seg_chunks * C
    int in_agg;
    const float* S0;
    const float* z0;
    int* dev_status;
    unsigned long long wait_ns;
    int force_timeout;
    KernelGammas g;
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

// Column sums of a [128 x DK] K-major swizzled bf16 tile (sum over its 128 rows)
// by 128 threads: thread t sums column pair (2 cp, 2 cp + 1), cp = t mod DK/2, over
// one of 256/DK row groups; a warp reads whole 128-byte rows (conflict-free).
// Partials go to `part` ([256/DK][DK] floats); the caller synchronises the 128
// threads and then reads colsum_total().
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

}  // namespace tck
}  // namespace la
