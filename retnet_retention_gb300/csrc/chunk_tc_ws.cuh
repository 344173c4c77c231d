// Chunkwise forward, warp-specialised tcgen05 pipeline (the output walk of a
// causal sequence or segment: mode kFull).
//
// The kernel template; chunk_tc_ws.cu instantiates it for the per-head decay,
// chunk_tc_ws_gated.cu for the per-token decay.
//
// Same arithmetic as the lockstep kernel in chunk_tc.cu ("Chunked Recurrent
// Representation", "RetNet" page; equations in chunk_tc.cu's header), but
// the roles run concurrently and hand work over through mbarriers:
//
//   warp 0      TMA producer: Q, K, V of chunk c into a ring of 2-4 stages
//   warp 1      MMA issuer (one thread): per chunk c, MMA4 and MMA3 as soon as
//               E3 of c and epilogue B have readied S and the tiles (the state
//               chain), then MMA1 of c+1 into the other of two TMEM score
//               buffers, then MMA2 of c once E1 has written P (with a single O
//               buffer MMA3 also waits for E2 of c-1, and MMA1 of c+1 goes
//               either last, or first where epilogue B rescales the tiles
//               after MMA1: then the rest waits for S and P together)
//   warps 2-9   epilogue A: per chunk, E3 first (bf16 copy of S for MMA3,
//               S *= gamma^L), then E1 (scores -> decay mask -> bf16 P back into
//               TMEM; the other order where MMA1 of c+1 goes first); two warps
//               per TMEM lane quarter, each on half of the columns
//   warps 10-13 epilogue B: the entry state, the xi/zeta row scalings, the
//               z update, and E2 (O of the previous chunk -> global, divided
//               by the normaliser)
//   warps 14-   phi = elu + 1 on the Q/K tiles as they land (8 warps for
//               64-wide Q/K and value blocks, else 2), up to a ring's depth
//               ahead of the tensor work; in the factored-decay build instead
//               V *= zeta (see FACT below)
//
// so that the state chain (MMA4 of c -> E3 of c+1 -> MMA4 of c+1) waits for
// nothing but E3 and epilogue B's per-chunk work, and E1, phi and E2 run beside
// it.  TMEM (512 columns): two score/P buffers at 0 and 128, O at 256 (two
// buffers for DVB = 64), S after O.
//
// The normaliser: z is one more value column ("Linear Attention" page, the
// normalised form; z_c = gamma^L z_{c-1} + sum_j zeta_j k^_j is S's recurrence
// for an all-ones value column).  With signed features the denominator can
// be a small difference of large sums, so no term of it is rounded to bf16:
// E1 takes the row sums of the scores in fp32 before P is rounded; for
// gamma = 1 MMA3 is issued with N = DVB + 16, the bf16 copy of S followed by a
// block holding z_{c-1} as a bf16 value and its bf16 residual in two columns,
// so O's columns DVB and DVB + 1 collect q^_i . z_{c-1} to about 16 bits; for
// gamma < 1 (where Q is scaled by xi in bf16 for MMA3) epilogue B takes
// xi_i q^_i . z_{c-1} in fp32 from the unscaled tile as it scales it.  z
// itself stays in fp32 shared memory, updated by decayed column sums of the
// unscaled K tile.
//
// Taken for DVB = 64 with any flags and for DVB = 128 without the
// normaliser; other cases use the lockstep kernel.
//
// Every wait is bounded; a role that times out raises a shared abort flag,
// every other role's waits then give up too, all roles meet at the end, the
// producer and issuer wait (bounded) for their own copies and MMAs, the CTA
// records LA_ERR_TIMEOUT and frees its TMEM.
#pragma once

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "chunk_tc_common.cuh"
#include "launch.h"
#include "trace.h"

// Development timeline (compiled only with -DLA_TIMELINE): CTA 0 stamps its SM's
// cycle counter at pipeline events into a device array the host reads back (the
// cycle counter: a read of the global timer costs far more than the events it
// would time).
#ifdef LA_TIMELINE
__device__ unsigned long long la_timeline[4096];
#define LA_TL(slot)                                                                        \
    do {                                                                                   \
        if (blockIdx.x == 0)                                                               \
            la_timeline[((slot) + (STATE_ONLY ? 2048 : 0)) & 4095] = (unsigned long long)clock64() | 1ull; \
    } while (0)
extern "C" __attribute__((visibility("default"))) int la_timeline_read(unsigned long long* host,
                                                                          int n) {
    if (n > 4096) n = 4096;
    return cudaMemcpyFromSymbol(host, la_timeline, (size_t)n * 8) == cudaSuccess ? n : -1;
}
__device__ unsigned long long la_cta_times[4 * 1024];  // per CTA: start, end (x2 kernels)
extern "C" __attribute__((visibility("default"))) int la_cta_times_read(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, la_cta_times, sizeof(la_cta_times)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int la_timeline_clear() {
    static const unsigned long long z2[4 * 1024] = {};
    cudaMemcpyToSymbol(la_cta_times, z2, sizeof(z2));
    static const unsigned long long zeros[4096] = {};
    return cudaMemcpyToSymbol(la_timeline, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -1;
}
#define LA_CTA_T(which)                                                                  \
    do {                                                                                 \
        if (threadIdx.x == 0 && blockIdx.x < 1024)                                       \
            la_cta_times[(STATE_ONLY ? 2048 : 0) + 2 * blockIdx.x + (which)] = la::tc::global_timer_ns(); \
    } while (0)
#else
#define LA_TL(slot) \
    do {            \
    } while (0)
#define LA_CTA_T(which) \
    do {                \
    } while (0)
#endif

namespace la {

using namespace tck;

namespace {

// Feature-map group: 8 warps for d_k = d_v-block = 64 with phi, else 2.  More
// warps hide the exp latency of phi; without phi they would only take registers
// (the SM's register file is split over its four schedulers: 704 threads get 80
// registers each, 512 get 128), and for the wider tiles the registers of the
// extra warps cost more than they give.
constexpr int threads_c(int dk, int dvb, bool phi) { return phi && dk == 64 && dvb == 64 ? 256 : 64; }
constexpr int threads_ws(int dk, int dvb, bool phi) { return 448 + threads_c(dk, dvb, phi); }
// The block size the compiler budgets registers for: for 64-wide tiles without
// phi the cap of a 640-thread block (96 registers) measured faster than the
// 128 that 512 threads would allow; the factored-decay build (fact) keeps 128.
constexpr int bound_ws(int dk, int dvb, bool phi, bool fact = false) {
    return !phi && !fact && dk == 64 && dvb == 64 ? 640 : threads_ws(dk, dvb, phi);
}
constexpr int kWgA = 2;   // first warp of epilogue A (8 warps: two per TMEM lane quarter)
constexpr int kWgB = 10;  // first warp of epilogue B
constexpr int kWgC = 14;  // first warp of the feature-map group
constexpr int kBarA = 1;  // named barrier ids
constexpr int kBarB = 2;
constexpr int kBarEntry = 3;  // epilogue B has put the entry state in TMEM (A + B)
constexpr int kBarC = 4;
constexpr int kBarP = 5;      // E1: the first column half has read its scores (A)
constexpr int kThreadsA = 256;
constexpr uint32_t kColScores = 0;  // + 128 * buffer
constexpr uint32_t kColO = 256;

constexpr uint32_t kSmemLimit = 232448;  // opt-in shared memory per CTA

// POS: the features are phi(.) > 0, so no term of the normaliser is negative.
// GATED: per-token decay; each stage also holds its chunk's cumulative log2
// decays and decays (2 x 128 fp32, after V).
template <int DK, int DVB, bool NORM, bool POS, bool GATED>
struct LayoutWS {
    static constexpr uint32_t kQ = (DK / 64) * kBlk;
    static constexpr uint32_t kK = (DK / 64) * kBlk;
    static constexpr uint32_t kV = (DVB / 64) * kBlk;
    static constexpr uint32_t oGate = kQ + kK + kV;     // within a stage
    static constexpr uint32_t kGate = GATED ? 2 * 128 * 4 : 0;
    static constexpr uint32_t kStage = kQ + kK + kV + kGate;  // a multiple of 1024
    // bf16 S, MN-major, 64-column blocks DK * 128 bytes apart; with the
    // normaliser one more block whose first 16 columns hold z
    static constexpr uint32_t kSB = (DVB / 64 + (NORM ? 1 : 0)) * (DK * 128);
    // positive features: a [128 x 64] block after V whose column 0 is ones (MMA2's
    // extra columns collect sum_j P_ij); signed features: fp32 row sums from E1 and,
    // for gamma < 1, xi_i q^_i . z_{c-1} from epilogue B
    static constexpr uint32_t kOnes = NORM && POS ? kBlk : 0;
    static constexpr uint32_t kDQ = NORM && !POS ? 2 * 128 * 4 : 0;      // by chunk parity
    static constexpr uint32_t kRS = NORM && !POS ? 3 * 2 * 128 * 4 : 0;  // 3 chunks x 2 halves
    static constexpr uint32_t kSmall = DK * 4 + 256 * 4 + kDQ + kRS + 32 * 8 + 16 + 1024;
    // ring depth: as many stages (up to 4) as shared memory holds
    static constexpr int NS = (4 * kStage + kSB + kOnes + kSmall <= kSmemLimit) ? 4
                            : (3 * kStage + kSB + kOnes + kSmall <= kSmemLimit) ? 3 : 2;
    static constexpr uint32_t oSB = NS * kStage;
    static constexpr uint32_t oOnes = oSB + kSB;        // 1024-byte aligned
    static constexpr uint32_t oZ = oOnes + kOnes;       // float z[DK]
    static constexpr uint32_t oZP = oZ + DK * 4;        // float colsum partials [256/DK][DK]
    static constexpr uint32_t oDQ = oZP + 256 * 4;      // float [2][128] (normaliser, gamma < 1)
    static constexpr uint32_t oRS = oDQ + kDQ;          // float [3][2][128] (normaliser)
    static constexpr uint32_t oBar = oRS + kRS;         // 32 mbarrier slots
    static constexpr uint32_t oFlags = oBar + 32 * 8;   // int abort, uint32 tmem slot
    static constexpr uint32_t kBytes = oFlags + 16;
    static constexpr uint32_t kAlloc = kBytes + 1024;   // slack for 1024-byte alignment
    // O accumulators: two for DVB = 64 (E2 of a chunk overlaps the next chunk's MMAs),
    // one for DVB = 128; then S.  With the normaliser an O accumulator has
    // DVB + 16 columns (column DVB: the denominator), its slot rounded up to 32.
    static constexpr int NOB = DVB == 64 ? 2 : 1;
    static constexpr int NO = NORM ? DVB + 16 : DVB;    // MMA2 (positive features) / MMA3 N
    static constexpr uint32_t kOSlot = (NO + 31) / 32 * 32;
    static constexpr uint32_t kColS = kColO + NOB * kOSlot;
    static_assert(kAlloc <= kSmemLimit, "shared memory budget");
    static_assert(kColS + DVB <= 512, "tensor memory budget");
    static_assert(!NORM || NOB == 2, "the normaliser's hand-overs assume two O buffers");
};

// Barriers.  Stage barriers (full, empty, qk) have one slot per ring stage;
// hand-overs that one side could otherwise complete twice before the other
// side waits once are double-buffered by chunk parity (sfull, sready, pready);
// o_full / o_empty cannot run ahead.  Per chunk c with two O buffers:
// sready(c) = the bf16 copy of S and the scaled S and tiles are in place for
// MMA3/MMA4 (epilogues A and B); pready(c) = P is in TMEM for MMA2 (epilogue A).
// With one O buffer and MMA1 of the next chunk issued first, pready(c) carries
// both (epilogues A and B).  sdone(c) =
// MMA3/MMA4 of c are complete; in a state walk sdone completes once, after the
// last MMA4.  A parity wait is sound only while its barrier is at most one phase
// behind the phase awaited: every wait here is placed so that it is.
enum Bars {
    kFull0 = 0, kEmpty0 = 4, kQk0 = 8, kReadyS0 = 12, kSfull0 = 16, kSfull1, kPready0, kPready1,
    kOfull0, kOfull1, kOempty0, kOempty1, kNever, kDrain, kSdone, kSready0, kSready1,
    kRsum0, kNumBars = kRsum0 + 3
};
static_assert(kNumBars <= 32, "mbarrier slots");

// STATE_ONLY: the walk of a segment's own state contribution (mode
// kStateOnly: K and V only, MMA4 only).  Its per-chunk hand-over to the
// issuer (kReadyS) has one slot per ring stage, which bounds how far the
// epilogues may run ahead.
//
// PHI: the launch applies phi (p.phi), which sizes the feature-map group and
// makes every term of the normaliser non-negative.
// GATED: a per-token decay a_t (p.gate) in place of the head's gamma: inside a
// chunk the powers of gamma become cumulative log-decays b_i = sum_{s<=i} log a_s
// ("Linear Attention, RWKV, and RetNet", 13.3 subsection 4, the gated decay):
// gamma^(i+1) -> 2^(b_i), gamma^(L-1-j) -> 2^(b_(L-1) - b_j), gamma^L ->
// 2^(b_(L-1)) (b in log2 units), and the score mask's running product steps by
// a_j instead of gamma.
// The kernel body: chunk_tc_ws_kernel runs one build, chunk_tc_ws_pick_kernel (the
// per-token decay) picks one of two per CTA.
template <int DK, int DVB, bool NORM, bool STATE_ONLY, bool PHI, bool GATED, bool FACT>
__device__ __forceinline__ void chunk_tc_ws_body(const TcParams& p) {
    static_assert(!FACT || (!PHI && !NORM), "the factored decay is for plain retention");
    static_assert(!(FACT && GATED && STATE_ONLY), "a state walk with per-token decays takes the row scalings");
    constexpr int kThreadsC = threads_c(DK, DVB, PHI);
    constexpr int kThreadsWS = threads_ws(DK, DVB, PHI);
    using Lay = LayoutWS<DK, DVB, NORM && !STATE_ONLY, PHI, GATED>;
    constexpr bool kOnesSum = NORM && PHI;   // sum_j P_ij through MMA2 and the ones block
    constexpr bool kE1Sum = NORM && !PHI;    // sum_j P_ij in fp32 from E1
    static_assert(!NORM || DVB == 64, "the normaliser's columns fit tensor memory only for DVB = 64");
    extern __shared__ __align__(1024) char smem_raw[];
    char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* zs = reinterpret_cast<float*>(sm + Lay::oZ);
    float* dqz = reinterpret_cast<float*>(sm + Lay::oDQ);
    float* rsb = reinterpret_cast<float*>(sm + Lay::oRS);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Lay::oFlags);
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + Lay::oFlags + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int unit = blockIdx.x;
    const int seg = unit % p.n_seg;
    const int dvb = (unit / p.n_seg) % p.n_dvb;
    const int bh = unit / (p.n_seg * p.n_dvb);
    const int h = bh % p.H;
    const int v0 = dvb * DVB;
    const float l2g = p.g.log2g[h];
    const float gam = p.g.gamma[h];
    const bool unit_gamma = !GATED && gam == 1.0f;
    // FACT: factored decay (per-head gamma < 1, no feature map, no normaliser, z not
    // carried; the host launches this build when every head qualifies).  With
    // zeta_j = gamma^(L-1-j) taken into V (by the feature-map group, as the tile
    // lands, while MMA1 already runs on the raw Q and K), the decayed scores times V
    // are
    //   sum_j (q_i . k_j) gamma^(i-j) v_j = gamma^(i+1-L) sum_j (q_i . k_j) zeta_j v_j,
    // the read-out gamma^(i+1) q_i S_{c-1} = gamma^(i+1-L) q_i (gamma^L S_{c-1}), and
    // the state's update sum_j zeta_j k_j v_j^T = K^T (zeta V); so the whole output
    // row is gamma^(i+1-L) (P V' + Q gamma^L S_{c-1})_i with P = Q K^T masked to
    // j <= i and V' = zeta V (MMA2 and MMA4 both read V'): E1 only masks, Q and K
    // are never rescaled, E3 copies gamma^L S (which MMA4 accumulates onto anyway)
    // and E2 applies the one per-row factor.  The factor gamma^(i+1-L) reaches gamma^(1-C), so this
    // form is taken only while gamma^(C-1) >= 2^-64 for every head (every product
    // stays far inside the float and bf16 ranges); smaller gammas keep the row
    // scalings.
    constexpr bool fact = FACT;
    // Reversed time (factored build only, p.rev): the same sums over s >= t, by the
    // mirror image of the chunk.  Chunk c's tiles start at row T - (c + 1) C and its
    // tile row r stands at position C - 1 - r of the chunk in the reversed sequence
    // (o_i = sum_{j>=i} (q_i . k_j) gamma^(j-i) v_j + gamma^(L-i) q_i S with i, j
    // counted from the chunk's first row and L the rows it holds), so every decay
    // exponent takes the mirrored row mrow(r), the mask keeps j >= i, and the rows
    // before row 0 (mrow(r) >= L) are the padding, read as zeros.
    const bool rev = FACT && p.rev;
    auto mrow = [&](int r) { return rev ? kC - 1 - r : r; };
    // Order of the work per chunk with one O buffer.  Where epilogue B rescales the
    // tiles after MMA1 (gamma < 1 without the factored form, per-token decays),
    // MMA1 of chunk c+1 goes before the MMAs of chunk c so that E1 and the
    // rescaling of c+1 overlap them, E1 goes before E3, and S and P hand over
    // together (kPready).  Otherwise nothing needs that overlap, and waiting for
    // chunk c+1's tiles first would put their load on every chunk's critical path
    // (a 96 KB stage, two in the ring): the MMAs of chunk c go first, then MMA1 of
    // c+1; E3 (released by MMA4 of c) goes before E1 (released by MMA1 of c+1) and
    // hands S over on its own (kSready), so MMA3 and MMA4 of c+1 run while E1
    // turns c+1's scores into P.  With two O buffers S and P always hand over apart.
    const bool mma1_first = Lay::NOB == 1 && !(fact || unit_gamma);
    const bool e3_first = Lay::NOB == 2 || !mma1_first;  // also: S and P hand over apart
    const int n_chunks = (p.T + kC - 1) / kC;
    const int cb = seg * p.seg_chunks;
    const int ce = min(n_chunks, cb + p.seg_chunks);
    const int n = ce - cb;  // chunks of this unit
    // Decay factors of a chunk.  With the per-token decay they come from the chunk's
    // cumulative log2 decays gc in its ring stage (read only after the stage's full
    // barrier); with gamma, gc is unused.
    auto gate_of = [&](int s) {
        return reinterpret_cast<const float*>(sm + s * Lay::kStage + Lay::oGate);
    };
    auto dec_xi = [&](const float* gc, int r) {  // row r of Q: gamma^(r+1)
        return GATED ? exp2f(gc[r]) : gamma_pow(l2g, (float)(r + 1));
    };
    auto dec_zeta = [&](const float* gc, int r, int L) {  // row r of K: gamma^(L-1-r), 0 past L
        return r < L ? (GATED ? exp2f(gc[L - 1] - gc[r]) : gamma_pow(l2g, (float)(L - 1 - r))) : 0.f;
    };
    auto dec_total = [&](const float* gc, int L) {  // the state's decay over the chunk: gamma^L
        return GATED ? exp2f(gc[L - 1]) : gamma_pow(l2g, (float)L);
    };
    // The factored build with the per-token decay takes its factors about the middle
    // exponent beta = (b_0 + b_(L-1)) / 2 of the chunk: zeta_j = 2^(beta - b_j) into V,
    // the row factor 2^(b_i - beta), and MMA3 and MMA4 work on 2^beta S_{c-1}, so that
    // TMEM holds S_c 2^(beta - b_(L-1)) after MMA4, a factor that the next chunk's E3 and
    // the exit state take out again.  Every factor stays within 2^(+-Delta/2) for a
    // chunk that decays by 2^-Delta from its first row to its last.
    auto fact_beta = [&](const float* gc, int L) { return 0.5f * (gc[0] + gc[L - 1]); };
    const uint64_t lim = p.wait_ns;
    if (tid == 0) LA_TL(4000);
    LA_CTA_T(0);
    griddep_launch_dependents();  // the next kernel's CTAs may be scheduled (it waits itself)

    constexpr int NS = Lay::NS;
    constexpr int NOB = Lay::NOB;
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&bar[b], 1);
        for (int q = 0; q < NS; ++q) mbar_init(&bar[kEmpty0 + q], 2);  // MMA commit + epilogue B
        mbar_init(&bar[kSready0], 2);  // epilogue A + epilogue B (S and P apart)
        mbar_init(&bar[kSready1], 2);
        // P ready: epilogue A alone where S and P hand over apart; else both here
        // (epilogue A + epilogue B)
        mbar_init(&bar[kPready0], e3_first ? 1 : 2);
        mbar_init(&bar[kPready1], e3_first ? 1 : 2);
        // state walk: epilogue B, plus epilogue A when S must be rescaled (gamma < 1)
        for (int q = 0; q < NS; ++q) mbar_init(&bar[kReadyS0 + q], unit_gamma ? 1 : 2);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&p.tmQ);
        prefetch_tensormap(&p.tmK);
        prefetch_tensormap(&p.tmV);
    }
    if (warp == 1) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    if constexpr (kOnesSum && !STATE_ONLY) {
        // the block after V for MMA2's extra columns: ones in column 0, zeros elsewhere
        // (read through the async proxy)
        for (int i = tid; i < (int)(kBlk / 16); i += kThreadsWS) {
            const uint32_t one = (i & 7) == ((i >> 3) & 7) ? 0x3F80u : 0u;  // logical piece 0 of row i >> 3
            reinterpret_cast<uint4*>(sm + Lay::oOnes)[i] = make_uint4(one, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t sbase = smem_addr(sm);
    if (tid == 0) LA_TL(4001);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;  // TMEM lane of this thread (epilogue warps)

    bool forced = false;
    if (p.force_timeout) {  // test hook: a wait on a barrier nothing arrives on
        if (tid == 0 && !mbar_wait(&bar[kNever], 0, lim)) record_status(p.dev_status, LA_ERR_TIMEOUT);
        forced = true;
    }

    // ---- entry state into TMEM and z into smem: epilogue B (all 128 lanes), at the
    // start of its role below, while the producer already loads the first chunks;
    // epilogue A waits for it (kBarEntry) before its first read of S.
    auto load_entry_state = [&]() {
        const int sidx = bh * p.in_nseg + seg;
        const bool has_in = p.S_in != nullptr && !STATE_ONLY;
        if (has_in && p.in_agg) {
            // entry state of segment `seg` from S0 and the contributions of segments
            // 0 .. seg-1 (at most kFoldMax - 1 of them), 8 columns at a time with
            // every contribution's loads issued before the recurrence runs over them
            // the state's decay over segment q: gamma^len, or 2^(the segment's total
            // log2 decay) with the per-token decay
            const float gs_all = GATED ? 0.f : gamma_pow(l2g, (float)(p.seg_chunks * kC));
            auto seg_decay = [&](int q) {
                return GATED ? exp2f(p.seg_l2[bh * p.in_nseg + q]) : gs_all;
            };
            const size_t seg_stride = (size_t)DK * p.dv;
            const int rr = row < DK ? row : 0;  // rows >= DK load nothing
            const float* arow = p.S_in + ((size_t)(bh * p.in_nseg) * DK + rr) * p.dv + v0;
            const float* s0row = p.S0 ? p.S0 + ((size_t)bh * DK + rr) * p.dv + v0 : nullptr;
            for (int c0 = 0; c0 < DVB; c0 += 32) {
                uint32_t r[32];
#pragma unroll
                for (int h8 = 0; h8 < 32; h8 += 8) {
                    float4 a[kFoldMax][2];
#pragma unroll
                    for (int q = 0; q < kFoldMax; ++q)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            a[q][e] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (row < DK) {
                                if (q == 0 && s0row)
                                    a[q][e] = *reinterpret_cast<const float4*>(s0row + c0 + h8 + 4 * e);
                                else if (q > 0 && q <= seg)
                                    a[q][e] = *reinterpret_cast<const float4*>(
                                        arow + (size_t)(q - 1) * seg_stride + c0 + h8 + 4 * e);
                            }
                        }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float4 x = a[0][e];
#pragma unroll
                        for (int q = 1; q < kFoldMax; ++q)
                            if (q <= seg) {
                                const float gs = seg_decay(q - 1);
                                x.x = fmaf(gs, x.x, a[q][e].x);
                                x.y = fmaf(gs, x.y, a[q][e].y);
                                x.z = fmaf(gs, x.z, a[q][e].z);
                                x.w = fmaf(gs, x.w, a[q][e].w);
                            }
                        r[h8 + 4 * e] = __float_as_uint(x.x);
                        r[h8 + 4 * e + 1] = __float_as_uint(x.y);
                        r[h8 + 4 * e + 2] = __float_as_uint(x.z);
                        r[h8 + 4 * e + 3] = __float_as_uint(x.w);
                    }
                }
                tmem_st32(tbase + lane_off + Lay::kColS + c0, r);
            }
            tmem_st_wait();
            if (row < DK) {
                float zz = p.z0 ? p.z0[(size_t)bh * DK + row] : 0.f;
                if (p.z_in)
                    for (int q = 0; q < seg; ++q)
                        zz = fmaf(seg_decay(q), zz, p.z_in[(size_t)(bh * p.in_nseg + q) * DK + row]);
                zs[row] = zz;
            }
            fence_before_sync();
            return;
        }
        const float* srow = has_in && row < DK ? p.S_in + ((size_t)sidx * DK + row) * p.dv + v0
                                               : nullptr;
        for (int c0 = 0; c0 < DVB; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (srow) x = *reinterpret_cast<const float4*>(srow + c0 + e);
                r[e] = __float_as_uint(x.x);
                r[e + 1] = __float_as_uint(x.y);
                r[e + 2] = __float_as_uint(x.z);
                r[e + 3] = __float_as_uint(x.w);
            }
            tmem_st32(tbase + lane_off + Lay::kColS + c0, r);
        }
        tmem_st_wait();
        if (row < DK) zs[row] = (has_in && p.z_in) ? p.z_in[(size_t)sidx * DK + row] : 0.f;
        fence_before_sync();
    };

    // per-role bookkeeping that the drain at the end needs
    int fills[4] = {0, 0, 0, 0};  // producer: TMA fills issued per stage
    if (tid == 0) LA_TL(4002);
    bool mma_issued = false;   // issuer: any MMA issued

    if (!forced && n > 0) {
        if (warp == 0 && lane == 0) {
            // ---------------- producer
            for (int it = 0; it < n; ++it) {
                const int s = it % NS;
                if (it >= NS &&
                    !mbar_wait_or_abort(&bar[kEmpty0 + s], ((it - NS) / NS) & 1, lim, abort_flag))
                    break;
                char* st = sm + s * Lay::kStage;
                const int y = rev ? p.T - (cb + it + 1) * kC : (cb + it) * kC;
                mbar_arrive_expect_tx(&bar[kFull0 + s],
                                      (STATE_ONLY ? Lay::kK + Lay::kV + Lay::kGate : Lay::kStage));
                if constexpr (GATED)
                    bulk_load(st + Lay::oGate, p.gate + ((size_t)bh * n_chunks + cb + it) * 256,
                              Lay::kGate, &bar[kFull0 + s]);
#pragma unroll
                for (int b = 0; b < DK / 64; ++b) {
                    if (!STATE_ONLY) tma_load_3d(st + b * kBlk, &p.tmQ, b * 64, y, bh, &bar[kFull0 + s]);
                    tma_load_3d(st + Lay::kQ + b * kBlk, &p.tmK, b * 64, y, bh, &bar[kFull0 + s]);
                }
#pragma unroll
                for (int b = 0; b < DVB / 64; ++b)
                    tma_load_3d(st + Lay::kQ + Lay::kK + b * kBlk, &p.tmV, v0 + b * 64, y, bh,
                                &bar[kFull0 + s]);
                ++fills[s];
                LA_TL(it * 16 + 0);
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer
            const uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
            // MMA2, with positive features plus the ones block's columns
            const uint32_t id_pv = idesc_bf16(128, kOnesSum ? Lay::NO : DVB, 0, 1);
            // MMA3, with the normaliser plus the z columns (for signed features and
            // gamma < 1 epilogue B takes xi_i q^_i . z_{c-1} in fp32 instead)
            const uint32_t id_qs = idesc_bf16(128, NORM && (PHI || unit_gamma) ? Lay::NO : DVB, 0, 1);
            const uint32_t id_kv = idesc_bf16(128, DVB, 1, 1);
            // descriptors of stage 0 and of bf16 S; the others are offsets from them
            const uint64_t dQk0 = smem_desc_sw128(sbase, 16, 1024);          // Q, K: K-major
            const uint64_t dKmn0 = smem_desc_sw128(sbase + Lay::kQ, kBlk, 1024);  // K: MN-major
            const uint64_t dSB = smem_desc_sw128(sbase + Lay::oSB, DK * 128, 1024);
            auto issue_mma1 = [&](int it) -> bool {
                const int s = it % NS;
                const uint32_t par = (it / NS) & 1;
                if (!mbar_wait_or_abort(&bar[kFull0 + s], par, lim, abort_flag)) return false;
                if (p.phi && !mbar_wait_or_abort(&bar[kQk0 + s], par, lim, abort_flag)) return false;
                fence_after_sync();
                const uint64_t dq = desc_adv(dQk0, s * Lay::kStage), dk = desc_adv(dq, Lay::kQ);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
                    mma_ss(tbase + kColScores + (it & 1) * 128, desc_adv(dq, off), desc_adv(dk, off),
                           id_qk, kk > 0);
                }
                mma_commit(&bar[kSfull0 + (it & 1)]);
                mma_issued = true;
                LA_TL(it * 16 + 1);
                return true;
            };
            if constexpr (STATE_ONLY) {
                for (int it = 0; it < n; ++it) {
                    const int s = it % NS;
                    if (!mbar_wait_or_abort(&bar[kReadyS0 + s], (it / NS) & 1, lim, abort_flag)) break;
                    fence_after_sync();
                    const uint64_t dk = desc_adv(dKmn0, s * Lay::kStage), dv = desc_adv(dk, Lay::kK);
#pragma unroll
                    for (int kk = 0; kk < kC / 16; ++kk)
                        mma_ss(tbase + Lay::kColS, desc_adv(dk, kk * 2048), desc_adv(dv, kk * 2048),
                               id_kv, 1u);
                    mma_commit(&bar[kOfull0]);
                    mma_commit(&bar[kEmpty0 + s]);
                    if (it == n - 1) mma_commit(&bar[kSdone]);  // the exit state is complete
                    mma_issued = true;
                    LA_TL(it * 16 + 3);
                }
                (void)issue_mma1;
                (void)id_pv;
                (void)id_qs;
            }
            // Per chunk, with two O buffers: MMA3/MMA4 as soon as S is ready (the state
            // chain), then MMA1 of the next chunk, then MMA2 once P is ready.  With one
            // O buffer MMA3 also waits for E2 of the previous chunk: either MMA1 of the
            // next chunk goes first and MMA3/MMA4/MMA2 follow once S and P are ready
            // (mma1_first), or MMA3/MMA4 go once S is ready, MMA2 once P is, and MMA1
            // of the next chunk last.
            bool ok = !STATE_ONLY && issue_mma1(0);
            for (int it = 0; it < n && ok; ++it) {
                const int s = it % NS;
                if (mma1_first && it + 1 < n && !(ok = issue_mma1(it + 1))) break;
                if (!mbar_wait_or_abort(&bar[(e3_first ? kSready0 : kPready0) + (it & 1)], (it >> 1) & 1,
                                        lim, abort_flag))
                    break;
                LA_TL(it * 16 + 2);
                const int ob = it % NOB;  // O buffer of this chunk
                if (it >= NOB &&
                    !mbar_wait_or_abort(&bar[kOempty0 + ob], ((it - NOB) / NOB) & 1, lim, abort_flag))
                    break;
                fence_after_sync();
                const uint32_t ocol = tbase + kColO + ob * Lay::kOSlot;
                const uint64_t dq = desc_adv(dQk0, s * Lay::kStage);
                const uint64_t dk = desc_adv(dKmn0, s * Lay::kStage), dv = desc_adv(dk, Lay::kK);
                // V for MMA2: its 64-column blocks are kBlk apart; with positive features
                // the ones block stands in for the next one (N = DVB + 16)
                const uint32_t va = sbase + s * Lay::kStage + Lay::kQ + Lay::kK;
                const uint64_t dv2 = kOnesSum ? smem_desc_sw128(va, sbase + Lay::oOnes - va, 1024) : dv;
                // MMA3: O = Q^ S_bf16 (K = DK)
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
                    mma_ss(ocol, desc_adv(dq, off), desc_adv(dSB, kk * 2048), id_qs, kk > 0);
                }
                // factored decay: V' = zeta V from the feature-map group (MMA4 and MMA2)
                if (FACT) {
                    if (!mbar_wait_or_abort(&bar[kQk0 + s], (it / NS) & 1, lim, abort_flag)) break;
                    fence_after_sync();
                }
                // MMA4: S += K^^T V (M = 128, rows >= DK unused; K = 128 tokens)
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ss(tbase + Lay::kColS, desc_adv(dk, kk * 2048), desc_adv(dv, kk * 2048), id_kv,
                           1u);
                mma_commit(&bar[kSdone]);
                if (NOB == 2 && it + 1 < n && !(ok = issue_mma1(it + 1))) break;
                if (e3_first) {
                    if (!mbar_wait_or_abort(&bar[kPready0 + (it & 1)], (it >> 1) & 1, lim, abort_flag))
                        break;
                    fence_after_sync();
                }
                // MMA2: O += P V (A = P from TMEM, K = 128 tokens)
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_ts(ocol, tbase + kColScores + (it & 1) * 128 + kk * 8, desc_adv(dv2, kk * 2048),
                           id_pv, 1u);
                mma_commit(&bar[kOfull0 + ob]);
                mma_commit(&bar[kEmpty0 + s]);
                LA_TL(it * 16 + 3);
                if (NOB == 1 && !mma1_first && it + 1 < n && !(ok = issue_mma1(it + 1))) break;
            }
        } else if (warp >= kWgA && warp < kWgB) {
            // ---------------- epilogue A: E1 (P) and E3 (S copies).  Warps kWgA..+3 take
            // the first half of the columns (half 0), warps kWgA+4..+7 the second.
            const int t = tid - kWgA * 32;
            const int half = t >> 7;
            named_bar_sync(kBarEntry, kThreadsA + 128);  // the entry state is in TMEM
            fence_after_sync();
            constexpr int kSHalf = DVB / 2;  // S columns per half
            if constexpr (STATE_ONLY) {
                // only S = gamma^L S before each MMA4 (nothing to do when gamma == 1)
                for (int it = 0; it < n && !unit_gamma; ++it) {
                    const int L = min(kC, p.T - (cb + it) * kC);
                    if (it >= 1 || GATED) {  // MMA4 of the previous chunk; the chunk's decays
                        bool ok = it < 1 || mbar_wait_or_abort(&bar[kOfull0], (it - 1) & 1, lim, abort_flag);
                        if (GATED && ok)
                            ok = mbar_wait_or_abort(&bar[kFull0 + it % NS], (it / NS) & 1, lim, abort_flag);
                        if (named_bar_or(kBarA, kThreadsA, !ok)) break;
                        fence_after_sync();
                    }
                    const float gL = dec_total(gate_of(it % NS), L);
                    for (int c0 = half * kSHalf; c0 < (half + 1) * kSHalf; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(tbase + lane_off + Lay::kColS + c0, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * gL);
                        tmem_st32(tbase + lane_off + Lay::kColS + c0, r);
                    }
                    tmem_st_wait();
                    fence_before_sync();
                    named_bar_sync(kBarA, kThreadsA);
                    if (t == 0) mbar_arrive(&bar[kReadyS0 + it % NS]);
                }
            }
            // Per chunk, E3 (S after MMA3/MMA4 of the previous chunk -> bf16 copy for
            // MMA3, S *= gamma^L before MMA4) and E1 (scores -> P for MMA2).  With two O
            // buffers E3 goes first and hands over on its own (kSready), so the state
            // chain does not wait for E1 (kPready).  With one, both hand over together
            // (kPready, after the second of the two); E1 goes first where MMA1 of the
            // chunk is issued before the previous chunk's MMAs (mma1_first: E1 then
            // overlaps them), else E3 does.
            float lc_prev = 0.f;  // factored, per-token decay: TMEM holds S_{c-1} 2^-lc_prev
            for (int it = 0; it < n && !STATE_ONLY; ++it) {
                const int c = cb + it;
                const int L = min(kC, p.T - c * kC);
                bool fail = false;
#pragma unroll
                for (int step = 0; step < 2; ++step) {
                    if (e3_first == (step == 0)) {  // ---- E3
                        if (it >= 1 || GATED) {  // MMA3/MMA4 of the previous chunk; the decays
                            bool ok = it < 1 || mbar_wait_or_abort(&bar[kSdone], (it - 1) & 1, lim, abort_flag);
                            if (GATED && ok)
                                ok = mbar_wait_or_abort(&bar[kFull0 + it % NS], (it / NS) & 1, lim, abort_flag);
                            if (named_bar_or(kBarA, kThreadsA, !ok)) { fail = true; break; }
                            fence_after_sync();
                            if (t == 0) LA_TL(it * 16 + 6);
                        }
                        float gL = unit_gamma ? 1.f : dec_total(gate_of(it % NS), L);
                        float gL2 = 1.f;
                        if constexpr (FACT && GATED) {
                            // 2^beta S_{c-1} from TMEM's S_{c-1} 2^-lc, as two factors (each
                            // >= 2^-80 in range; their product need not be)
                            const float* gc = gate_of(it % NS);
                            const float beta = fact_beta(gc, L);
                            gL = exp2f(lc_prev);
                            gL2 = exp2f(beta);
                            lc_prev = gc[L - 1] - beta;
                        }
#pragma unroll
                        for (int c0 = half * kSHalf; c0 < (half + 1) * kSHalf; c0 += 32) {
                            uint32_t rs[32];
                            tmem_ld32(tbase + lane_off + Lay::kColS + c0, rs);
                            tmem_ld_wait();
                            if (fact) {  // MMA3 reads gamma^L S_{c-1}
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    rs[e] = __float_as_uint(GATED ? __uint_as_float(rs[e]) * gL * gL2
                                                                  : __uint_as_float(rs[e]) * gL);
                            }
                            if (row < DK) {
#pragma unroll
                                for (int e8 = 0; e8 < 32; e8 += 8) {
                                    const int v = c0 + e8;
                                    uint4 wv;
                                    wv.x = pack_bf16x2(__uint_as_float(rs[e8 + 0]), __uint_as_float(rs[e8 + 1]));
                                    wv.y = pack_bf16x2(__uint_as_float(rs[e8 + 2]), __uint_as_float(rs[e8 + 3]));
                                    wv.z = pack_bf16x2(__uint_as_float(rs[e8 + 4]), __uint_as_float(rs[e8 + 5]));
                                    wv.w = pack_bf16x2(__uint_as_float(rs[e8 + 6]), __uint_as_float(rs[e8 + 7]));
                                    *reinterpret_cast<uint4*>(sm + Lay::oSB + (v >> 6) * (DK * 128) +
                                                              sw128_offset(row, v & 63)) = wv;
                                }
                            }
                            if (!unit_gamma) {
                                if (!fact) {
#pragma unroll
                                    for (int e = 0; e < 32; ++e) rs[e] = __float_as_uint(__uint_as_float(rs[e]) * gL);
                                }
                                tmem_st32(tbase + lane_off + Lay::kColS + c0, rs);
                            }
                        }
                        if (!unit_gamma) tmem_st_wait();
                        fence_proxy_async_smem();
                        fence_before_sync();
                        named_bar_sync(kBarA, kThreadsA);
                        if (t == 0)  // S alone (E3 first), or S and P together (E3 second)
                            mbar_arrive(&bar[(e3_first ? kSready0 : kPready0) + (it & 1)]);
                        if (t == 0) LA_TL(it * 16 + 7);
                    } else {  // ---- E1
                        bool ok1 = mbar_wait_or_abort(&bar[kSfull0 + (it & 1)], (it >> 1) & 1, lim, abort_flag);
                        if (GATED && ok1)  // the chunk's decays
                            ok1 = mbar_wait_or_abort(&bar[kFull0 + it % NS], (it / NS) & 1, lim, abort_flag);
                        if (named_bar_or(kBarA, kThreadsA, !ok1)) { fail = true; break; }
                        fence_after_sync();
                        if (t == 0) LA_TL(it * 16 + 4);
                        const uint32_t sc = tbase + lane_off + kColScores + (it & 1) * 128;
                        const int i = row;
                        float rsum = 0.f;  // fp32 row sum of this half's scores (normaliser)
                        if constexpr (FACT) {
                            // the scores need only the causal mask (the decay is in V or is 1):
                            // both pieces loaded at once, one wait, then packed and stored.
                            // Pieces wholly on the masked side of the diagonal are P = 0 for
                            // the whole warp (above it; below it in reversed time).
                            const int lq = warp & 3, pa = 2 * half;
                            const bool za = rev ? pa < lq : pa > lq, zb = rev ? pa + 1 < lq : pa + 1 > lq;
                            uint32_t ra[32], rb[32];
                            if (!za) tmem_ld32(sc + 32 * pa, ra);
                            if (!zb) tmem_ld32(sc + 32 * pa + 32, rb);
                            tmem_ld_wait();
                            if (t == 0) LA_TL(it * 16 + 15);
                            if (half == 0) {
                                fence_before_sync();
                                named_bar_arrive(kBarP, kThreadsA);
                            }
                            // one piece of P: columns j0 .. j0 + 31 kept where j <= i (j >= i
                            // in reversed time), two instantiations so that neither form
                            // tests the direction per element
                            auto pack_piece = [&](const uint32_t* r, int j0, bool z, uint32_t* pk, auto dir) {
                                constexpr bool kRev = decltype(dir)::value;
#pragma unroll
                                for (int e = 0; e < 32; e += 2) {
                                    const int j = j0 + e;
                                    const bool k0 = kRev ? j >= i : j <= i;
                                    const bool k1 = kRev ? j + 1 >= i : j + 1 <= i;
                                    pk[e >> 1] = z ? 0u
                                                   : pack_bf16x2(k0 ? __uint_as_float(r[e]) : 0.f,
                                                                 k1 ? __uint_as_float(r[e + 1]) : 0.f);
                                }
                            };
                            auto pack = [&](const uint32_t* r, int j0, bool z, uint32_t* pk) {
                                if (rev)
                                    pack_piece(r, j0, z, pk, BoolC<true>{});
                                else
                                    pack_piece(r, j0, z, pk, BoolC<false>{});
                            };
                            uint32_t pk[16];
                            pack(ra, 32 * pa, za, pk);
                            if (half == 1) {
                                named_bar_sync(kBarP, kThreadsA);
                                fence_after_sync();
                            }
                            tmem_st16(sc + 16 * pa, pk);
                            pack(rb, 32 * pa + 32, zb, pk);
                            tmem_st16(sc + 16 * pa + 16, pk);
                        } else {
                            // this half's two 32-column pieces of scores, one at a time.  P (bf16
                            // pairs) goes to columns [0, 64): half 1's P lands on half 0's second
                            // piece, so half 1 stores only after half 0 has read that piece (kBarP).
                            // A warp's 32 rows and a piece's 32 columns are the same 32 x 32 block
                            // for every lane, so a piece above the diagonal is P = 0 for the whole
                            // warp (no load), and only the piece on the diagonal needs the mask
                            // j <= i.
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const int c0 = 64 * half + 32 * q;
                                const int pq = c0 >> 5, lq = warp & 3;
                                // (in the 80-register phi build the skip spills a few registers
                                // and still saves about 3 % of the walk)
                                const bool zero = pq > lq;
                                uint32_t r[32];
                                if (!zero) {
                                    tmem_ld32(sc + c0, r);
                                    tmem_ld_wait();
                                }
                                if (half == 0 && q == 1) {
                                    fence_before_sync();
                                    named_bar_arrive(kBarP, kThreadsA);
                                }
                                uint32_t pk[16];
                                if (zero) {
#pragma unroll
                                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                                } else {
                                    // gamma^(i-j) by a running product from the piece's top column down
                                    const int jt = min(i, c0 + 31);
                                    float w = unit_gamma || fact ? 1.f : gamma_pow(l2g, (float)(i - jt));
                                    const bool diag = pq == lq;
                                    if constexpr (GATED) {
                                        // 2^(b_i - b_j), stepping down a column by a_j (the decay
                                        // of token j); the per-head code below is kept apart: the
                                        // two forms of the loop compile differently enough to
                                        // matter for the 80-register build
                                        const float* gc = gate_of(it % NS);
                                        const float* ga = gc + 128;
                                        w = exp2f(gc[i] - gc[jt]);
#pragma unroll
                                        for (int e = 30; e >= 0; e -= 2) {
                                            float x1 = __uint_as_float(r[e + 1]), x0 = __uint_as_float(r[e]);
                                            const bool in1 = c0 + e + 1 <= i, in0 = c0 + e <= i;
                                            x1 = in1 ? x1 * w : 0.f;
                                            if (in1) w *= ga[c0 + e + 1];
                                            x0 = in0 ? x0 * w : 0.f;
                                            if (in0) w *= ga[c0 + e];
                                            if (kE1Sum) rsum += x1 + x0;
                                            pk[e >> 1] = pack_bf16x2(x0, x1);
                                        }
                                    } else if constexpr (!PHI) {  // each pair packed as soon as it is scaled
#pragma unroll
                                        for (int e = 30; e >= 0; e -= 2) {
                                            float x1 = __uint_as_float(r[e + 1]), x0 = __uint_as_float(r[e]);
                                            if (!unit_gamma && !fact) {
                                                x1 *= w;
                                                if (!diag || c0 + e + 1 <= i) w *= gam;
                                                x0 *= w;
                                                if (!diag || c0 + e <= i) w *= gam;
                                            }
                                            if (diag) {
                                                x1 = c0 + e + 1 <= i ? x1 : 0.f;
                                                x0 = c0 + e <= i ? x0 : 0.f;
                                            }
                                            if (kE1Sum) rsum += x1 + x0;
                                            pk[e >> 1] = pack_bf16x2(x0, x1);
                                        }
                                    } else {  // (the form that fits 80 registers)
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
                                        for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(a[e], a[e + 1]);
                                    }
                                }
                                if (half == 1 && q == 0) {
                                    named_bar_sync(kBarP, kThreadsA);
                                    fence_after_sync();
                                }
                                tmem_st16(sc + (c0 >> 1), pk);
                            }
                        }
                        // the row sums before rounding P: with signed features the
                        // denominator can be a small difference of large sums, which the
                        // bf16 P would not resolve.  To E2 through shared memory, one slot
                        // per chunk, three slots (E1 of chunk c + 3 waits for MMA1 of c + 3,
                        // which the issuer starts only after E2 of c has freed c's O buffer)
                        if (kE1Sum) rsb[(it % 3) * 256 + half * 128 + row] = rsum;
                        tmem_st_wait();
                        if (e3_first) {  // E1 second: P on its own
                            fence_before_sync();
                            named_bar_sync(kBarA, kThreadsA);
                            if (t == 0) {
                                mbar_arrive(&bar[kPready0 + (it & 1)]);
                                if (kE1Sum) mbar_arrive(&bar[kRsum0 + it % 3]);
                            }
                        }
                        if (t == 0) LA_TL(it * 16 + 5);
                    }
                }
                if (fail) break;
            }
        } else if (warp >= kWgC) {
            // ---------------- feature map: phi on Q and K (K only for a state walk), rows
            // past the end zeroed, then release the stage to the issuer (kQk); with the
            // factored decay instead V *= zeta (Q and K stay as they are)
            const int t = tid - kWgC * 32;
            // factored decay: zeta of this thread's rows (t >> 3) + (kThreadsC / 8) m, as
            // bf16 pairs, for the chunk length zL (recomputed only when it changes)
            constexpr int kRowsC = 1024 / kThreadsC;
            uint32_t zh[kRowsC], zl[kRowsC];
            int zL = -1;
            for (int it = 0; it < n && (p.phi || fact); ++it) {
                const int s = it % NS;
                const int L = min(kC, p.T - (cb + it) * kC);
                bool ok = mbar_wait_or_abort(&bar[kFull0 + s], (it / NS) & 1, lim, abort_flag);
                if (named_bar_or(kBarC, kThreadsC, !ok)) break;
                char* st = sm + s * Lay::kStage;
                if (t == 0) LA_TL(it * 16 + 12);
                if constexpr (FACT) {
                    if (GATED || L != zL) {  // (per-token decay: every chunk its own zeta)
                        const float* gc = GATED ? gate_of(s) : nullptr;
                        const float beta = GATED ? fact_beta(gc, L) : 0.f;
#pragma unroll
                        for (int m = 0; m < kRowsC; ++m) {
                            const int r = mrow((t >> 3) + (kThreadsC / 8) * m);
                            split_bf16x2(GATED ? (r < L ? exp2f(beta - gc[r]) : 0.f) : dec_zeta(nullptr, r, L),
                                         zh[m], zl[m]);
                        }
                        zL = L;
                    }
                    scale_rows_hl<DVB / 64, kThreadsC>(st + Lay::kQ + Lay::kK, zh, zl, t);
                } else if constexpr (STATE_ONLY && kThreadsC % 128 == 0) {  // all loads first
                    char* const tiles[1] = {st + Lay::kQ};
                    phi_rows_all<1, DK / 64, kThreadsC>(tiles, L, t);
                } else if constexpr (STATE_ONLY) {
                    phi_rows(st + Lay::kQ, DK / 64, L, t, kThreadsC);
                } else {  // one piece at a time, leaving the pipe to the epilogues' packs
                    phi_rows(st, DK / 64, L, t, kThreadsC);
                    phi_rows(st + Lay::kQ, DK / 64, L, t, kThreadsC);
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarC, kThreadsC);
                if (t == 0) mbar_arrive(&bar[kQk0 + s]);
                if (t == 0) LA_TL(it * 16 + 13);
            }
        } else if (warp >= kWgB) {
            // ---------------- epilogue B: entry state, scalings, z, E2
            const int t = tid - kWgB * 32;
            griddep_wait();  // entry states come from the previous kernel in the stream
            load_entry_state();
            named_bar_arrive(kBarEntry, kThreadsA + 128);
            int L_prev = 0;
            float rho_prev = 1.f;
            float lc_last = 0.f;  // factored, per-token decay: TMEM holds S 2^-lc_last
            bool stop = false;
            // exit state: S (after the last MMA4, which the caller has waited for) and z
            auto write_exit_state = [&]() {
                if (!p.S_out) return;
                const bool write = !p.out_last_only || seg == p.n_seg - 1;
                const int oidx = bh * p.out_nseg + (p.out_last_only ? 0 : seg);
                for (int c0 = 0; c0 < DVB; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + Lay::kColS + c0, r);
                    tmem_ld_wait();
                    if constexpr (FACT && GATED) {
                        const float f = exp2f(lc_last);
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                    }
                    if (write && row < DK) {
                        float* srow = p.S_out + ((size_t)oidx * DK + row) * p.dv + v0 + c0;
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(srow + e) =
                                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
                    }
                }
                if (write && p.z_out && dvb == 0 && row < DK) p.z_out[(size_t)oidx * DK + row] = zs[row];
            };
            // E2 of chunk `it`: O rows -> global, divided by the normaliser
            // rho: the factored build's row factor 2^(b_i - beta) with the per-token decay
            // (read from the chunk's stage while it was held)
            auto do_e2 = [&](int it, int L, float rho) -> bool {
                bool ok = mbar_wait_or_abort(&bar[kOfull0 + it % NOB], (it / NOB) & 1, lim, abort_flag);
                if (kE1Sum && ok) ok = mbar_wait_or_abort(&bar[kRsum0 + it % 3], (it / 3) & 1, lim, abort_flag);
                if (named_bar_or(kBarB, 128, !ok)) return false;
                fence_after_sync();
                if (t == 0) LA_TL(it * 16 + 10);
                const uint32_t ocol = tbase + lane_off + kColO + (it % NOB) * Lay::kOSlot;
                float inv = 1.f;
                if (NORM) {  // sum_j P_ij + xi_i q^_i . z_{c-1}
                    // O's columns DVB and DVB + 1: MMA3's z block (z_{c-1} and its residual)
                    // and, with positive features, MMA2's ones column (sum_j P_ij)
                    float den = 0.f;
                    if (PHI || unit_gamma) {
                        den = __uint_as_float(tmem_ld1(ocol + DVB)) + __uint_as_float(tmem_ld1(ocol + DVB + 1));
                        tmem_ld_wait();
                    }
                    if (kE1Sum) {
                        den += rsb[(it % 3) * 256 + row] + rsb[(it % 3) * 256 + 128 + row];
                        if (!unit_gamma) den += dqz[(it & 1) * 128 + row];
                    }
                    inv = 1.f / norm_den(den, p.normalize, p.eps);
                }
                if (fact) inv = GATED ? rho : gamma_pow(l2g, (float)(mrow(row) + 1 - L));  // gamma^(i+1-L)
                const int c = cb + it;
                // the row's place in the sequence (reversed time: chunk c starts at row
                // T - (c + 1) C, before row 0 for the last chunk); rows past the chunk's
                // L are padding and store nothing
                const int trow = rev ? p.T - (c + 1) * kC + row : c * kC + row;
                const bool live = mrow(row) < L;
                __nv_bfloat16* orow = p.O + ((size_t)bh * p.T + (size_t)max(trow, 0)) * p.dv + v0;
                // 64 columns a round in the factored build with 128 registers a thread
                // (two loads, one wait), else 32.  The O buffer is released once the
                // last round is in registers; in the factored build the earlier
                // round's values are packed (bf16) and held until then, so the
                // release waits for no store.
                constexpr int kW = FACT && bound_ws(DK, DVB, PHI, FACT) <= 512 ? 2 : 1;  // 32-column loads a round
                constexpr int kRounds = DVB / (32 * kW);
                constexpr int kHold = kW == 2 ? kRounds - 1 : 0;  // rounds held packed
                uint32_t held[kHold > 0 ? kHold : 1][16 * kW];
                // 16 kW words = 32 kW columns of the row: 32-byte stores where O is
                // 32-byte aligned (each a whole sector), else 16-byte ones; O is not
                // allocated in L1 and is first to leave L2 (nothing here reads it back)
                const uint64_t opol = l2_evict_first_policy();
                auto store_packed = [&](const uint32_t* pk, int col) {
                    if (p.o_align32) {
#pragma unroll
                        for (int e = 0; e < 16 * kW; e += 8) st_global_v8(orow + col + 2 * e, pk + e, opol);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16 * kW; e += 4)
                            st_global_v4(orow + col + 2 * e, pk[e], pk[e + 1], pk[e + 2], pk[e + 3], opol);
                    }
                };
#pragma unroll
                for (int rd = 0; rd < kRounds; ++rd) {
                    uint32_t r[kW][32];
#pragma unroll
                    for (int hf = 0; hf < kW; ++hf) tmem_ld32(ocol + 32 * (kW * rd + hf), r[hf]);
                    tmem_ld_wait();
                    if (rd == kRounds - 1) {
                        fence_before_sync();
                        named_bar_sync(kBarB, 128);
                        if (t == 0) mbar_arrive(&bar[kOempty0 + it % NOB]);
                        if (t == 0) LA_TL(it * 16 + 14);
                    }
                    uint32_t pk[16 * kW];
#pragma unroll
                    for (int hf = 0; hf < kW; ++hf)
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            pk[16 * hf + (e >> 1)] =
                                pack_bf16x2(__uint_as_float(r[hf][e]) * inv, __uint_as_float(r[hf][e + 1]) * inv);
                    if (rd < kHold) {
#pragma unroll
                        for (int e = 0; e < 16 * kW; ++e) held[rd][e] = pk[e];
                        continue;
                    }
                    if (live) {
#pragma unroll
                        for (int h = 0; h < kHold; ++h) store_packed(held[h], 32 * kW * h);
                        store_packed(pk, 32 * kW * rd);
                    }
                }
                if (t == 0) LA_TL(it * 16 + 11);
                return true;
            };
            if constexpr (STATE_ONLY) {
                float lam = 0.f;  // per-token decay: the segment's total log2 decay (thread 0)
                for (int it = 0; it < n; ++it) {
                    const int s = it % NS;
                    const int L = min(kC, p.T - (cb + it) * kC);
                    char* tK = sm + s * Lay::kStage + Lay::kQ;
                    // the tile, and phi(K) from the feature-map group
                    bool ok = mbar_wait_or_abort(&bar[kFull0 + s], (it / NS) & 1, lim, abort_flag);
                    if (ok && (p.phi || fact))  // phi(K), or zeta V, from the feature-map group
                        ok = mbar_wait_or_abort(&bar[kQk0 + s], (it / NS) & 1, lim, abort_flag);
                    if (named_bar_or(kBarB, 128, !ok)) {
                        stop = true;
                        break;
                    }
                    const float* gc = gate_of(s);
                    const float gL = unit_gamma ? 1.f : dec_total(gc, L);  // read while the stage is ours
                    if (GATED && t == 0) lam += gc[L - 1];
                    // z_c = gamma^L z_{c-1} + sum_j zeta_j phi(K)[j], the sums in fp32 from the
                    // unscaled tile: with gamma < 1 in the pass that scales K, with gamma = 1
                    // (no scaling) beside MMA4
                    float* zpart = reinterpret_cast<float*>(sm + Lay::oZP);
                    // K^ = zeta . phi(K), rows >= L zeroed (here unless the feature-map
                    // group took zeta into V); then MMA4 may go (kReadyS)
                    if (!unit_gamma && !fact) {
                        auto zeta = [&](int r) { return dec_zeta(gc, r, L); };
                        if (p.track_z) {
                            scale_rows_zsum<DK>(tK, zeta, zpart, t);
                        } else {
#pragma unroll 1
                            for (int b = 0; b < DK / 64; ++b)  // one 64-column block at a time
                                scale_rows_all<1, 128>(tK + b * kBlk, zeta, t);
                        }
                    }
                    fence_proxy_async_smem();
                    fence_before_sync();
                    named_bar_sync(kBarB, 128);
                    if (t == 0) mbar_arrive(&bar[kReadyS0 + s]);
                    if (p.track_z) {
                        if (unit_gamma) {
                            colsum_partial<DK>(tK, t, zpart);
                            named_bar_sync(kBarB, 128);
                        }
                        if (t < DK) zs[t] = fmaf(gL, zs[t], colsum_total<DK>(zpart, t));
                    }
                    // every read of the stage was before the last barrier (the next chunk's
                    // partials are written only after its first barrier)
                    if (t == 0) mbar_arrive(&bar[kEmpty0 + s]);
                    if (t == 0) LA_TL(it * 16 + 9);
                }
                if (!stop && !*abort_flag) {
                    // the last MMA4 on a barrier of its own: this role runs up to a ring of
                    // stages ahead of the MMAs, so o_full may be two or more phases behind
                    // here, and a parity wait would then return for an earlier phase
                    bool ok = mbar_wait_or_abort(&bar[kSdone], 0, lim, abort_flag);
                    if (!named_bar_or(kBarB, 128, !ok)) {
                        fence_after_sync();
                        write_exit_state();
                        if (GATED && t == 0 && dvb == 0 && p.seg_l2)
                            p.seg_l2[bh * p.out_nseg + seg] = lam;
                    }
                }
                stop = true;
            }
            for (int it = 0; it < n && !stop; ++it) {
                const int s = it % NS;
                const int c = cb + it;
                const int L = min(kC, p.T - c * kC);
                char* tQ = sm + s * Lay::kStage;
                char* tK = tQ + Lay::kQ;
                // The tiles of this chunk (phi's writes to them are visible through kQk);
                // with gamma < 1 they are scaled in place, so MMA1 must be done with the
                // unscaled ones first
                bool ok = unit_gamma || fact
                              ? mbar_wait_or_abort(&bar[kFull0 + s], (it / NS) & 1, lim, abort_flag)
                              : mbar_wait_or_abort(&bar[kSfull0 + (it & 1)], (it >> 1) & 1, lim, abort_flag);
                if (ok && p.phi) ok = mbar_wait_or_abort(&bar[kQk0 + s], (it / NS) & 1, lim, abort_flag);
                if (GATED && ok)  // the chunk's decays
                    ok = mbar_wait_or_abort(&bar[kFull0 + s], (it / NS) & 1, lim, abort_flag);
                if (named_bar_or(kBarB, 128, !ok)) break;
                if (t == 0) LA_TL(it * 16 + 8);
                const float* gc = GATED ? gate_of(s) : nullptr;
                // the chunk's decay of z, read while the stage is ours (per-token decay)
                const float gL_gated = GATED ? dec_total(gc, L) : 0.f;
                float rho = 1.f;
                if constexpr (FACT && GATED) {
                    const float beta = fact_beta(gc, L);
                    rho = exp2f(gc[row] - beta);
                    lc_last = gc[L - 1] - beta;
                }
                // z_c = gamma^L z_{c-1} + sum_j zeta_j phi(K)[j], the sums in fp32 from the
                // unscaled tile: with gamma = 1 while epilogue B would otherwise wait for
                // MMA3 of the previous chunk, with gamma < 1 in the pass that scales K
                float* zpart = reinterpret_cast<float*>(sm + Lay::oZP);
                const bool zsum = NORM || p.track_z;
                if (unit_gamma) {
                    if (zsum) colsum_partial<DK>(tK, t, zpart);
                } else if (!fact) {  // (factored decay: nothing to scale here)
                    auto xi = [&](int r) { return dec_xi(gc, r); };
                    auto zeta = [&](int r) { return dec_zeta(gc, r, L); };
                    if (kE1Sum)  // and xi_i q^_i . z_{c-1} from the unscaled tile, for E2
                        scale_rows_dot<DK>(tQ, xi, zs, dqz + (it & 1) * 128, t);
                    else
                        row_pass(tQ, DK / 64, false, xi, t, 128);
                    if (zsum)
                        scale_rows_zsum<DK>(tK, zeta, zpart, t);
                    else
                        row_pass(tK, DK / 64, false, zeta, t, 128);
                    fence_proxy_async_smem();
                }
                if (NORM && (PHI || unit_gamma)) {
                    // z_{c-1} into the block after bf16 S, once MMA3 of the previous chunk
                    // has read the old one; MMA3 then adds xi_i q^_i . z_{c-1} to O's columns
                    // DVB and DVB + 1
                    if (it >= 1) {
                        ok = mbar_wait_or_abort(&bar[kSdone], (it - 1) & 1, lim, abort_flag);
                        if (named_bar_or(kBarB, 128, !ok)) break;
                    }
                    if (t < DK) {
                        // z in two bf16 columns, its rounding and the residual, so q^ . z
                        // keeps about 16 bits even when its terms cancel
                        const float zf = zs[t];
                        const __nv_bfloat16 zh = __float2bfloat16_rn(zf);
                        const __nv_bfloat16 zl = __float2bfloat16_rn(zf - __bfloat162float(zh));
                        const uint32_t zw = (uint32_t)__bfloat16_as_ushort(zh) |
                                            ((uint32_t)__bfloat16_as_ushort(zl) << 16);
                        char* zb = sm + Lay::oSB + (DVB / 64) * (DK * 128);
                        *reinterpret_cast<uint4*>(zb + sw128_offset(t, 0)) = make_uint4(zw, 0u, 0u, 0u);
                        *reinterpret_cast<uint4*>(zb + sw128_offset(t, 8)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                fence_before_sync();
                named_bar_sync(kBarB, 128);  // tiles scaled, z block written, z sums stored
                if (t == 0) mbar_arrive(&bar[(e3_first ? kSready0 : kPready0) + (it & 1)]);
                if (zsum && t < DK) {
                    const float gL = unit_gamma ? 1.f : GATED ? gL_gated : gamma_pow(l2g, (float)L);
                    zs[t] = fmaf(gL, zs[t], colsum_total<DK>(zpart, t));
                }
                if (t == 0) mbar_arrive(&bar[kEmpty0 + s]);  // our generic reads of stage s are done
                if (t == 0) LA_TL(it * 16 + 9);
                if (it >= 1 && !do_e2(it - 1, L_prev, rho_prev)) {
                    stop = true;
                    break;
                }
                L_prev = L;
                rho_prev = rho;
            }
            if (!STATE_ONLY && !stop && !*abort_flag) {
                if (do_e2(n - 1, L_prev, rho_prev)) write_exit_state();  // do_e2 waited for MMA4
            }
        }
    }

    __syncwarp();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (*abort_flag || forced) {
        record_status(p.dev_status, LA_ERR_TIMEOUT);
        if (warp == 0 && lane == 0) {  // our own TMA fills must land before the smem is released
            for (int s = 0; s < NS; ++s)
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
    if (warp == 1) tmem_dealloc(tbase, 512);
    if (tid == 0) LA_TL(4003);
    LA_CTA_T(1);
}

template <int DK, int DVB, bool NORM, bool STATE_ONLY, bool PHI, bool GATED, bool FACT>
__global__ void __launch_bounds__(bound_ws(DK, DVB, PHI, FACT), 1) chunk_tc_ws_kernel(const __grid_constant__ TcParams p) {
    chunk_tc_ws_body<DK, DVB, NORM, STATE_ONLY, PHI, GATED, FACT>(p);
}

// Per-token decay, output walk without normaliser or z: the CTA takes the factored
// build when every chunk of its unit keeps its decay from first row to last at or
// above 2^-160 (p.gate_flags, from gate_prep_kernel), else the row scalings.  Every
// warp reads the unit's flags and reaches the same answer.
template <int DK, int DVB>
__global__ void __launch_bounds__(bound_ws(DK, DVB, false, true), 1) chunk_tc_ws_pick_kernel(const __grid_constant__ TcParams p) {
    const int unit = blockIdx.x;
    const int seg = unit % p.n_seg;
    const int bh = unit / (p.n_seg * p.n_dvb);
    const int n_chunks = (p.T + kC - 1) / kC;
    const int cb = seg * p.seg_chunks;
    const int ce = min(n_chunks, cb + p.seg_chunks);
    int bad = 0;
    for (int c = cb + (int)(threadIdx.x & 31); c < ce; c += 32) bad |= p.gate_flags[(size_t)bh * n_chunks + c];
    if (__any_sync(0xffffffffu, bad))
        chunk_tc_ws_body<DK, DVB, false, false, false, true, false>(p);
    else
        chunk_tc_ws_body<DK, DVB, false, false, false, true, true>(p);
}

// pdl: launch as a programmatic dependent of the previous kernel in the stream
// (the kernel's entry-state reads wait for that kernel; everything else may
// start early).
template <int DK, int DVB, bool NORM, bool STATE_ONLY, bool PHI, bool GATED, bool FACT = false>
cudaError_t launch_ws(const TcParams& prm, int grid, cudaStream_t s, bool pdl) {
    using Lay = LayoutWS<DK, DVB, NORM && !STATE_ONLY, PHI, GATED>;
    auto kern = chunk_tc_ws_kernel<DK, DVB, NORM, STATE_ONLY, PHI, GATED, FACT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::kAlloc);
    if (e != cudaSuccess) return e;
    TraceScope trace(STATE_ONLY ? "chunk_tc_ws_kernel/state" : "chunk_tc_ws_kernel/full", s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads_ws(DK, DVB, PHI));
    cfg.dynamicSmemBytes = Lay::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, prm);
#ifdef LA_DEBUG_LAUNCH
    {  // development aid: the reason a launch was refused, with the kernel's resources
        cudaFuncAttributes fa;
        cudaFuncGetAttributes(&fa, kern);
        std::fprintf(stderr,
                     "launch_ws<%d,%d,%d,%d,%d,%d,%d>: %s; regs %d, local %zu B, max threads %d, "
                     "dynamic smem %u B, static smem %zu B, grid %d x %d\n",
                     DK, DVB, (int)NORM, (int)STATE_ONLY, (int)PHI, (int)GATED, (int)FACT,
                     cudaGetErrorString(e), fa.numRegs,
                     fa.localSizeBytes, fa.maxThreadsPerBlock, Lay::kAlloc, fa.sharedSizeBytes, grid,
                     threads_ws(DK, DVB, PHI));
    }
#endif
    return e;
}

template <int DK, int DVB>
cudaError_t launch_ws_pick(const TcParams& prm, int grid, cudaStream_t s, bool pdl) {
    using Lay = LayoutWS<DK, DVB, false, false, true>;
    auto kern = chunk_tc_ws_pick_kernel<DK, DVB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::kAlloc);
    if (e != cudaSuccess) return e;
    TraceScope trace("chunk_tc_ws_kernel/full", s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads_ws(DK, DVB, false));
    cfg.dynamicSmemBytes = Lay::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

// The kernel for the launch's shape, flags and decay.  Kernels with phi are
// instantiated apart where phi changes the kernel: the feature-map group of
// 64-wide tiles, and the normaliser's row sums.
template <bool GATED>
cudaError_t dispatch_ws(int dk, int dvb, bool normalize, const TcParams& prm, int grid,
                        cudaStream_t s, bool pdl) {
    const bool phi = prm.phi != 0;
    if (prm.fact) {  // plain retention with its decays in the factored form's range
        if (phi || normalize) return cudaErrorInvalidValue;
        const bool st = prm.mode == kStateOnly;
        if constexpr (GATED) {  // output walks, each CTA picking its build (a state walk
                                // with these decays keeps the row scalings)
            if (st) return cudaErrorInvalidValue;
            if (dk == 64 && dvb == 64) return launch_ws_pick<64, 64>(prm, grid, s, pdl);
            if (dk == 64 && dvb == 128) return launch_ws_pick<64, 128>(prm, grid, s, pdl);
            if (dk == 128 && dvb == 64) return launch_ws_pick<128, 64>(prm, grid, s, pdl);
            return cudaErrorInvalidValue;  // (no room for the decays beside two 96 KB stages at 128 x 128)
        } else {
            if (dk == 64 && dvb == 64)
                return st ? launch_ws<64, 64, false, true, false, false, true>(prm, grid, s, pdl)
                          : launch_ws<64, 64, false, false, false, false, true>(prm, grid, s, pdl);
            if (dk == 64 && dvb == 128)
                return st ? launch_ws<64, 128, false, true, false, false, true>(prm, grid, s, pdl)
                          : launch_ws<64, 128, false, false, false, false, true>(prm, grid, s, pdl);
            if (dk == 128 && dvb == 64)
                return st ? launch_ws<128, 64, false, true, false, false, true>(prm, grid, s, pdl)
                          : launch_ws<128, 64, false, false, false, false, true>(prm, grid, s, pdl);
            if (dk == 128 && dvb == 128)
                return st ? launch_ws<128, 128, false, true, false, false, true>(prm, grid, s, pdl)
                          : launch_ws<128, 128, false, false, false, false, true>(prm, grid, s, pdl);
            return cudaErrorInvalidValue;
        }
    }
    if (prm.mode == kStateOnly) {
        if (dk == 64 && dvb == 64)
            return phi ? launch_ws<64, 64, false, true, true, GATED>(prm, grid, s, pdl)
                       : launch_ws<64, 64, false, true, false, GATED>(prm, grid, s, pdl);
        if (dk == 64 && dvb == 128) return launch_ws<64, 128, false, true, false, GATED>(prm, grid, s, pdl);
        if (dk == 128 && dvb == 64) return launch_ws<128, 64, false, true, false, GATED>(prm, grid, s, pdl);
        if constexpr (!GATED)  // (no room for the per-token decays beside two 96 KB stages)
            if (dk == 128 && dvb == 128) return launch_ws<128, 128, false, true, false, false>(prm, grid, s, pdl);
        return cudaErrorInvalidValue;
    }
    if (normalize) {
        if (dk == 64 && dvb == 64)
            return phi ? launch_ws<64, 64, true, false, true, GATED>(prm, grid, s, pdl)
                       : launch_ws<64, 64, true, false, false, GATED>(prm, grid, s, pdl);
        if (dk == 128 && dvb == 64)
            return phi ? launch_ws<128, 64, true, false, true, GATED>(prm, grid, s, pdl)
                       : launch_ws<128, 64, true, false, false, GATED>(prm, grid, s, pdl);
        return cudaErrorInvalidValue;
    }
    if (dk == 64 && dvb == 64)
        return phi ? launch_ws<64, 64, false, false, true, GATED>(prm, grid, s, pdl)
                   : launch_ws<64, 64, false, false, false, GATED>(prm, grid, s, pdl);
    if (dk == 64 && dvb == 128) return launch_ws<64, 128, false, false, false, GATED>(prm, grid, s, pdl);
    if (dk == 128 && dvb == 64) return launch_ws<128, 64, false, false, false, GATED>(prm, grid, s, pdl);
    if constexpr (!GATED)
        if (dk == 128 && dvb == 128) return launch_ws<128, 128, false, false, false, false>(prm, grid, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace la
