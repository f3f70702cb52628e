// Backward pass: gradients recomputed tile by tile from the saved LSE.
//
// Method (johe.ru "Flash Attention: ...", section "Стадии вычисления", pass 2:
// the gradients are computed from the same tiles without storing the N x N
// matrix; "Проблема 3": keeping that matrix for the backward would double the
// memory).  With P = exp(scale S - LSE) rebuilt from the forward's LSE:
//     dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic,
//     dS = P o (dP - D),   dK = scale dS^T Q,   dQ = scale dS K.
//
// Three launches on one stream:
//   bwd_pre   D_i = rowsum(dO o O) in fp32 (one warp per row).
//   bwd_dkdv  work item = one 128-key tile (KV-tile parallel), taken by
//             persistent CTAs (one per SM): K_j, V_j stay in shared memory
//             for the item, Q_i / dO_i stream through a 2-stage ring;
//             tcgen05: S^T = K Q^T and dP^T = V dO^T into TMEM; S^T is read
//             out at once (so S^T of the next query tile can be issued while
//             P waits in registers); once dP^T is read, P^T and dS^T are
//             written over it as bf16 for dV += P^T dO and dK += dS^T Q, both
//             with A from TMEM; dK, dV accumulate in TMEM over all query
//             tiles.
//   bwd_dq    work item = one 128-query tile (Q-tile parallel), taken by
//             persistent CTAs: Q_i, dO_i are written into TMEM by the compute
//             threads and stay for the item; K_j / V_j
//             stream; S = Q K^T and dP = dO V^T take Q, dO from TMEM; dQ +=
//             dS K with dS from TMEM.  dQ is accumulated in fp32 TMEM and
//             written once, so the backward needs no atomics and is
//             deterministic.
// In both, one thread per TMEM lane (the 128 rows of the tile) computes P
// and dS for the 64 columns of its warpgroup; P stays in registers (packed
// bf16) so the next score MMA can be issued while dS is being formed.
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct Bwd {
    static constexpr int KCH = D / 64;
    static constexpr int TILE = 128 * D * 2;  // one 128-row bf16 tile
    static constexpr int CHUNK = 128 * 128;   // 128 rows x 128 bytes (one swizzle column block)
    static constexpr int OFF_FIXED = 0;       // two resident tiles
    static constexpr int OFF_STAGE = 2 * TILE;  // 2 stages x 2 streamed tiles
    static constexpr int OFF_VEC = OFF_STAGE + 4 * TILE;  // dkdv: lse2/delta per stage (2 x 1 KB)
    static constexpr int OFF_BAR = OFF_VEC + 2048;
    static constexpr int NBAR = 16;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16;  // the dynamic shared array is declared 1024-aligned
    // warps 0-7 compute (two warpgroups), 8 producer, 9 MMA issuer; the dK/dV pass adds warp 10,
    // a second issuer: there one thread cannot issue MMAs as fast as the tensor pipe runs them
    // while eight warps load the SM
    static constexpr int THREADS_DQ = 320, THREADS_DKDV = 352;
    static constexpr int PRODUCER = 8, MMA = 9, MMA2 = 10;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_A = 0;      // S / S^T fp32
    static constexpr uint32_t COL_B = 128;    // dP / dP^T fp32; dS (dQ pass) or P^T and dS^T (dK/dV pass) bf16 over it
    static constexpr uint32_t COL_ACC0 = 256; // dV (dkdv) or dQ (dq)
    static constexpr uint32_t COL_ACC1 = 256 + D;  // dK (dkdv)
    static constexpr uint32_t IDESC_SS = idesc_bf16(128, 128, 0, 0);
    static constexpr uint32_t IDESC_TS = idesc_bf16(128, D, 0, 1);
};

struct BwdParams {
    const __nv_bfloat16* q;   // the dQ pass loads its Q and dO rows straight into TMEM
    const __nv_bfloat16* dO;
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    const float* lse;
    const float* delta;
    int BH, Nq, Nk, causal, n_qt, n_kt;
    int window;  // > 0: causal sliding window of this many keys
    const int* lens_q;  // per-sequence query / key counts, or null (Nq / Nk)
    const int* lens_k;
    int H;
    int hc_kv, hc_q;  // heads per scheduling chunk of the dK/dV and dQ grids
    int n_pt;         // key-tile pairs per head (CTA-pair dK/dV grid)
    int hc_fu;        // heads per scheduling chunk of the single-pass grid
    float* dqacc;     // single pass: fp32 dQ accumulator [BH, Nq, D]
    float scale, scale_log2;
    DevError* err;
    uint64_t timeout_ns;
};

constexpr float kLog2e = 1.4426950408889634f;

// CTA order of a grid of BH heads x n_t tiles, tile 0 the longest: heads come
// in chunks of hc whose streamed operands fit in L2 together; within a chunk
// every head's tile 0 first, then every head's tile 1, and so on, so the
// hardware starts the longest CTAs first and the last wave is short ones.
__device__ __forceinline__ void chunked_order(int idx, int n_t, int BH, int hc, int& bh, int& t) {
    const int chunk_sz = hc * n_t;
    const int c = idx / chunk_sz;
    const int r = idx - c * chunk_sz;
    const int h0 = c * hc;
    const int hn = min(hc, BH - h0);
    t = r / hn;
    bh = h0 + (r - t * hn);
}

// Query and key counts of head bh's sequence (per-sequence lengths clamped to
// [0, Nq] and [0, Nk]; the forward records lengths out of range).  Rows and
// keys past them are padding: their LSE reads as -inf (P = 0), key columns are
// masked, and their gradients are stored as zeros.
__device__ __forceinline__ void bwd_seqlen(const BwdParams& p, int bh, int& nq, int& nk) {
    nq = p.Nq;
    nk = p.Nk;
    if (p.lens_q) nq = min(max(__ldg(p.lens_q + bh / p.H), 0), p.Nq);
    if (p.lens_k) nk = min(max(__ldg(p.lens_k + bh / p.H), 0), p.Nk);
}

// ------------------------------------------------------------------ D = rowsum(dO o O)
// HBM-bound: D/8 lanes per row, 16-byte loads, each warp with 2 row groups'
// loads in flight before it reduces (twice the CTAs of 4 groups, a shorter last
// wave: 26.5 -> 24.5 us at B=1, H=32, N=8192 with O and dO in L2, 33 -> 31 us
// from HBM).
template <int D>
constexpr int kPreRowsPerBlock = 8 * (32 / (D / 8)) * 2;

template <int D>
__global__ void __launch_bounds__(256)
bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
               float* __restrict__ delta, float* __restrict__ dqacc, long long rows) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, STEPS = 2;
    // the dK/dV pass launched after this grid may set up (and load K, V) meanwhile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // launched as a programmatic dependent of the kernel before it: O and dO may come from that
    // kernel, and D may still be read by it (the dQ pass of an earlier backward)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row0 = (long long)blockIdx.x * kPreRowsPerBlock<D> + (long long)warp * RPW * STEPS + lane / LPR;
    const int part = lane % LPR;
    uint4 x[STEPS], y[STEPS];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const long long row = row0 + st * RPW;
        x[st] = y[st] = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows) {
            x[st] = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
            y[st] = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + part);
        }
    }
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&x[st]);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&y[st]);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 u = __bfloat1622float2(a2[i]), v = __bfloat1622float2(b2[i]);
            sum = fmaf(u.x, v.x, sum);
            sum = fmaf(u.y, v.y, sum);
        }
#pragma unroll
        for (int w = LPR / 2; w >= 1; w >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, w);
        const long long row = row0 + st * RPW;
        if (part == 0 && row < rows) delta[row] = sum;
        // the single-pass backward accumulates dQ in fp32 here: every row starts at zero
        if (dqacc && row < rows) {
            float4* z = reinterpret_cast<float4*>(dqacc + row * D + part * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Issue C[tmem] = A B^T over K = D with both operands K-major 128-row tiles.
// The single issuing thread spends a few instructions per MMA: one descriptor
// of each operand per call, constant offsets per k-step, fixed accumulate flags.
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint32_t sA, uint32_t sB) {
    const uint64_t a0 = sdesc_sw128(sA, 16, 1024), b0 = sdesc_sw128(sB, 16, 1024);
    mma_ss_first(d_tmem, a0, b0, Bwd<D>::IDESC_SS);
#pragma unroll
    for (int k = 1; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * Bwd<D>::CHUNK + (k & 3) * 32;
        mma_ss_acc(d_tmem, sdesc_add(a0, off), sdesc_add(b0, off), Bwd<D>::IDESC_SS);
    }
}

// Issue C[tmem] (+)= A[tmem, 128 x 128 bf16] B[smem, 128 x D, MN-major].  The
// two compute warpgroups write the bf16 A operand in two halves, K = 0..63 at
// columns a_tmem + [0, 32) and K = 64..127 at a_tmem + [64, 96), each over the
// fp32 columns that warpgroup has itself already read (the dK/dV pass puts P^T
// at a_tmem = COL_B and dS^T at a_tmem = COL_B + 32, filling both halves).
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB, bool acc) {
    const uint64_t b0 = sdesc_sw128(sB, Bwd<D>::CHUNK, 1024);
    mma_ts(d_tmem, a_tmem, b0, Bwd<D>::IDESC_TS, acc ? 1u : 0u);
#pragma unroll
    for (int k = 1; k < 8; ++k)
        mma_ts_acc(d_tmem, a_tmem + k * 8 + (k >= 4 ? 32 : 0), sdesc_add(b0, k * 2048), Bwd<D>::IDESC_TS);
}

// Issue C[tmem] = A[tmem, 128 x D bf16] B^T with B a K-major 128-row tile in
// shared memory (the score products of the dQ pass: Q or dO from TMEM).
template <int D>
__device__ __forceinline__ void issue_ts_k(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB) {
    const uint64_t b0 = sdesc_sw128(sB, 16, 1024);
    mma_ts(d_tmem, a_tmem, b0, Bwd<D>::IDESC_SS, 0u);
#pragma unroll
    for (int k = 1; k < D / 16; ++k)
        mma_ts_acc(d_tmem, a_tmem + k * 8, sdesc_add(b0, (k >> 2) * Bwd<D>::CHUNK + (k & 3) * 32),
                   Bwd<D>::IDESC_SS);
}

// Writes columns [c0, c0 + D/2) of a 128-row accumulator row (thread = row)
// scaled by `mul` as bf16; each compute warpgroup stores its half.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, __nv_bfloat16* dst, float mul, bool valid,
                                              bool zero, int c0) {
    taddr += c0;
    dst += c0;
    const bool wide = ((uintptr_t)dst & 31) == 0;  // the same for every row: rows are 32-byte multiples
    constexpr int NQ = D / 64;  // 32-column chunks of this warpgroup's half
    uint32_t v[NQ][32];
    if (!zero) {  // (warp-uniform) every chunk's load in flight before the one wait
#pragma unroll
        for (int q4 = 0; q4 < NQ; ++q4) tmem_ld32_async(taddr + q4 * 32, v[q4]);
#pragma unroll
        for (int q4 = 0; q4 < NQ; ++q4) tmem_wait_ld(v[q4]);
    } else {
#pragma unroll
        for (int q4 = 0; q4 < NQ; ++q4)
#pragma unroll
            for (int i = 0; i < 32; ++i) v[q4][i] = 0u;
    }
#pragma unroll
    for (int q4 = 0; q4 < NQ; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16(__uint_as_float(v[q4][2 * i]) * mul, __uint_as_float(v[q4][2 * i + 1]) * mul);
        if (valid) store_row64(dst + q4 * 32, pk, wide);
    }
}

// Shared prologue: barriers, TMEM.  Returns the TMEM base.  A CTA pair
// allocates its columns collectively (one warp of each CTA) and both CTAs'
// barriers are initialised before either uses the other's.
template <int D, bool PAIR = false>
__device__ __forceinline__ uint32_t bwd_setup(uint8_t* smem, uint32_t bar0, const WaitCtl& ctl,
                                              const uint32_t* counts, int nbar) {
    const int tid = threadIdx.x, warp = tid >> 5;
    uint32_t* tmem_slot = (uint32_t*)(smem + Bwd<D>::OFF_MISC);
    if (tid == 0) {
        *ctl.abort = 0;
        for (int b = 0; b < nbar; ++b) mbar_init(bar0 + 8 * b, counts[b]);
        fence_mbar_init();
        if ((smem_u32(smem) & 1023u) != 0) record_error(ctl, kErrTimeout, kSiteAlign, 0);
    }
    if (warp == Bwd<D>::MMA) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), Bwd<D>::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), Bwd<D>::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    return *tmem_slot;
}

// Every wait of the kernel is bounded, so every thread of both CTAs of a pair
// arrives here; the collective free follows the last use of either CTA's TMEM.
template <int D, bool PAIR = false>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == Bwd<D>::MMA) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem, Bwd<D>::TMEM_COLS);
        else
            tmem_dealloc(tmem, Bwd<D>::TMEM_COLS);
    }
}

template <bool PAIR>
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const WaitCtl& ctl, int site) {
    if constexpr (PAIR)
        return mbar_wait_cl(bar, parity, ctl, site);
    else
        return mbar_wait(bar, parity, ctl, site);
}
template <bool PAIR>
__device__ __forceinline__ bool bdrain(uint32_t bar, uint32_t parity, const WaitCtl& ctl, int site) {
    if constexpr (PAIR)
        return mbar_drain_cl(bar, parity, ctl, site);
    else
        return mbar_drain(bar, parity, ctl, site);
}
// A commit of the issuing thread: in a pair it arrives on both CTAs' copies of `bar`.
template <bool PAIR>
__device__ __forceinline__ void bcommit(uint32_t bar) {
    if constexpr (PAIR)
        mma_commit_pair(bar);
    else
        mma_commit(bar);
}

// The pair's score products: A = this CTA's K (or V) tile, 128 keys x D; B = its
// 64 query rows of Q (or dO) in two 64-feature quadrants (X0, X1), one M = 256
// product over both CTAs.
constexpr uint32_t kQuad = 64 * 128;  // one 64-row x 64-feature bf16 quadrant, 8 KB
template <int D>
__device__ __forceinline__ void issue_ss_pair(uint32_t d_tmem, uint32_t sA, uint32_t sB) {
    constexpr uint32_t ID = idesc_bf16(256, 128, 0, 0);
    const uint64_t a0 = sdesc_sw128(sA, 16, 1024), b0 = sdesc_sw128(sB, 16, 1024);
    mma2_ss_first(d_tmem, a0, b0, ID);
#pragma unroll
    for (int k = 1; k < D / 16; ++k)
        mma2_ss_acc(d_tmem, sdesc_add(a0, (k >> 2) * Bwd<D>::CHUNK + (k & 3) * 32),
                    sdesc_add(b0, (k >> 2) * kQuad + (k & 3) * 32), ID);
}
// The pair's dV / dK products: A = P^T or dS^T from this CTA's TMEM (as in
// issue_ts); B = this CTA's 64-feature half of dO (or Q) over all 128 queries
// (quadrants Y0, Y1, back to back, MN-major): N = D over both CTAs.
template <int D>
__device__ __forceinline__ void issue_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint32_t sY, bool acc) {
    constexpr uint32_t ID = idesc_bf16(256, D, 0, 1);
    const uint64_t b0 = sdesc_sw128(sY, 2 * kQuad, 1024);
    mma2_ts(d_tmem, a_tmem, b0, ID, acc ? 1u : 0u);
#pragma unroll
    for (int k = 1; k < 8; ++k) mma2_ts_acc(d_tmem, a_tmem + k * 8 + (k >= 4 ? 32 : 0), sdesc_add(b0, k * 2048), ID);
}

// ------------------------------------------------------------------ dK, dV (KV-tile parallel)
// PAIR (d = 128): the two CTAs of a cluster take key tiles 2t and 2t + 1 of a
// head and run every product as one M = 256 tcgen05.mma (cta_group::2) issued
// by the even CTA.  Each CTA keeps its own K, V tile (A of the score products,
// its 128 of the 256 rows) and loads, per query tile, the parts of Q and dO
// that the products take from it as B.  The score products S^T = K Q^T and
// dP^T = V dO^T split B by query rows (rank r: queries 64r..64r+63, all
// features); dV += P^T dO and dK += dS^T Q split it by features (rank r:
// features 64r..64r+63, all queries).  So each CTA stages four 64 x 64
// quadrants of each operand: X0, X1 (its query rows, feature halves 0 and 1)
// and Y0, Y1 (its feature half, query rows 0-63 and 64-127); per k-step a
// product reads 2 KB of B from its shared memory instead of 4 KB.  The
// barriers the issuing thread waits on are the even CTA's (the odd CTA's loads
// and arrivals reach them through the cluster); its commits arrive on both
// CTAs' copies.  The loop runs over the query tiles either key tile sees; a
// tile one key tile does not see is masked out for it (P = 0).
template <int D, bool PAIR>
__global__ void __launch_bounds__(Bwd<D>::THREADS_DKDV, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const BwdParams p) {
    static_assert(!PAIR || D == 128, "CTA pairs at d = 128");
    using C = Bwd<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;  // 1024-aligned (checked in bwd_setup)
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    // barriers
    // S: S^T ready; SF: S^T read out of TMEM (the next S^T may overwrite it); DP: dP^T ready;
    // DS: P^T and dS^T written over dP^T (bf16, TMEM)
    // STE[s]: stage s free, once both issuers' products that read it are done (two arrivals);
    // TD, TD2: teardown of issuer 1 and 2; ACC: an item's dK and dV complete
    // KE, VE: an item's K (its last S^T) and V (its last dP^T) no longer read; ACCE: its dK, dV
    // read out of TMEM
    const uint32_t B_KV = bar0, B_STF = bar0 + 8, B_STE = bar0 + 24, B_S = bar0 + 40, B_DP = bar0 + 48,
                   B_DS = bar0 + 56, B_ACC = bar0 + 64, B_TD = bar0 + 72, B_SF = bar0 + 80, B_TD2 = bar0 + 88,
                   B_KE = bar0 + 96, B_ACCE = bar0 + 104, B_VE = bar0 + 112, B_VF = bar0 + 120;
    // STF: the producer's 32 lanes (of each CTA of a pair); SF, DS: every compute thread, or in a
    // pair one elected thread per compute warp of each CTA; ACCE: every compute thread
    constexpr uint32_t N_STF = PAIR ? 64 : 32, N_SD = PAIR ? 16 : 256;
    const uint32_t counts[16] = {1, N_STF, N_STF, 2, 2, 1, 1, N_SD, 1, 1, N_SD, 1, 1, 256, 1, 1};
    static_assert(16 <= C::NBAR, "barrier space");
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const uint32_t tmem = bwd_setup<D, PAIR>(smem, bar0, ctl, counts, 16);
    const uint32_t rank = PAIR ? cluster_rank() : 0u;
    const bool lead = rank == 0;  // the CTA whose thread issues the products
    // a barrier the issuing thread waits on, as addressed from this CTA
    auto lead_bar = [&](uint32_t b) { return PAIR ? mapa_shared(b, 0) : b; };
    auto arrive_lead = [&](uint32_t b) {
        if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(b, 0));
        else
            mbar_arrive(b);
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Work items: key tiles (in a pair, key-tile pairs) in the chunked order (key tile 0, the most
    // query tiles when causal, first; heads in L2-sized chunks).  A single CTA is persistent
    // (next_chunked_item) and, while its compute warps store one item's dK and dV, already loads
    // the next item's K, V and first query tiles and runs its first score products.  A pair
    // takes the one item of its cluster.
    const int n_items = PAIR ? p.n_pt * p.BH : p.n_kt * p.BH;
    const int chunk_items = p.hc_kv * p.n_kt;
    auto next_item = [&](ItemSeq& q) -> int {
        if constexpr (PAIR)
            return q.rd++ == 0 ? (int)(blockIdx.x >> 1) : n_items;
        else
            return next_chunked_item(q, n_items, chunk_items, gridDim.x, blockIdx.x, p.causal != 0);
    };
    struct Item {
        int bh, kt, nq, nk, off, i0, n;  // n query tiles from i0 (the union of a pair's two key tiles)
    };
    auto item_of = [&](int w) {
        Item it;
        if constexpr (PAIR) {
            int pt;
            chunked_order(w, p.n_pt, p.BH, p.hc_kv, it.bh, pt);
            it.kt = 2 * pt + (int)rank;
        } else {
            chunked_order(w, p.n_kt, p.BH, p.hc_kv, it.bh, it.kt);
        }
        bwd_seqlen(p, it.bh, it.nq, it.nk);
        it.off = it.nk - it.nq;
        const int kt_lo = it.kt - (int)rank, kt_hi = PAIR ? kt_lo + 1 : it.kt;  // the key tiles sharing the loop
        it.i0 = 0;
        if (p.causal) {
            const int first_q = kt_lo * 128 - it.off;  // smallest query that sees key kt_lo*128
            it.i0 = first_q <= 0 ? 0 : first_q / 128;
        }
        auto tile_end = [&](int t) {  // one past the last query tile that sees key tile t
            int e = t * 128 < it.nk ? (it.nq + 127) / 128 : 0;  // no query tile past the sequence
            if (p.window > 0) {  // the last query that sees the tile's last key
                const long long qlast = (long long)t * 128 + 127 - it.off + p.window - 1;
                e = qlast < 0 ? 0 : (int)min((long long)e, qlast / 128 + 1);
            }
            return e;
        };
        const int i_end = max(tile_end(kt_lo), tile_end(kt_hi));
        it.n = it.i0 < i_end ? i_end - it.i0 : 0;
        return it;
    };
    const uint32_t sK = s_base + C::OFF_FIXED, sV = sK + C::TILE;
    auto sQ = [&](int st) { return s_base + C::OFF_STAGE + st * 2 * C::TILE; };
    auto sDO = [&](int st) { return s_base + C::OFF_STAGE + st * 2 * C::TILE + C::TILE; };
    float* vec = (float*)(smem + C::OFF_VEC);  // stage s: lse2 at [s*256], delta at [s*256 + 128]
    // K (completing B_KV) and V (B_VF) load separately: an item's K is free after its last S^T,
    // its V only after its last dP^T, and the next item's first S^T needs only K
    auto load_t = [&](const Item& it, bool is_v) {  // one lane
        const uint32_t bar = is_v ? B_VF : B_KV;
        if (lead) mbar_arrive_expect_tx(bar, (PAIR ? 2 : 1) * C::TILE);
        const uint32_t fb = lead_bar(bar);
        const uint32_t dst = is_v ? sV : sK;
        const CUtensorMap* m = is_v ? &map_v : &map_k;
        for (int c = 0; c < C::KCH; ++c) {
            if constexpr (PAIR)
                tma_load_3d_pair(dst + c * C::CHUNK, m, fb, c * 64, it.kt * 128, it.bh, l2_policy_evict_last());
            else
                tma_load_3d(dst + c * C::CHUNK, m, fb, c * 64, it.kt * 128, it.bh, l2_policy_evict_last());
        }
    };
    auto load_kv = [&](const Item& it) {
        load_t(it, false);
        load_t(it, true);
    };
    // the first item's K and V do not come from the preprocess: they load before the wait for it
    ItemSeq q0;
    const int w_first = next_item(q0);
    const bool first_active = w_first < n_items && item_of(w_first).n > 0;
    int k_fills = 0, v_fills = 0;  // K and V loads issued (producer lane 0)
    if (warp == C::PRODUCER && lane == 0 && first_active && !*abort_flag) {
        load_kv(item_of(w_first));
        k_fills = v_fills = 1;
    }
    // Launched as a programmatic dependent of the preprocess, this grid may start before D is
    // complete: every read of D comes after this wait.  Then the dQ pass launched after this grid
    // (which reads D too) may start on SMs this grid leaves free.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Every role counts the query tiles (g) and the items with at least one (a) it has taken:
    // the per-tile barriers complete once per query tile, B_KV, B_VF, B_ACC, B_KE, B_VE and B_ACCE once
    // per item with query tiles, so their parities follow these counts.
    if (warp == C::PRODUCER) {
        // ------------------------------------------------------------ producer (whole warp)
        uint32_t issued = 0, issued_par = 0;
        if (!*abort_flag) {
            const uint64_t pol = l2_policy_evict_last();
            if (lane == 0) {
                tma_prefetch_desc(&map_q);
                tma_prefetch_desc(&map_do);
            }
            // per-column LSE*log2(e) and D of query tile i (4 values of each per lane),
            // read from global memory one tile ahead so the load latency is off the
            // path from "stage free" to "TMA issued"
            float nl2[4], ndl[4];
            auto fetch_vec = [&](const Item& it, int i) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int q = i * 128 + lane + 32 * t;
                    nl2[t] = INFINITY;
                    ndl[t] = 0.f;
                    if (q < it.nq) {
                        const float L = p.lse[(size_t)it.bh * p.Nq + q];
                        nl2[t] = (L == -INFINITY) ? INFINITY : L * kLog2e;
                        ndl[t] = p.delta[(size_t)it.bh * p.Nq + q];
                    }
                }
            };
            bool ok = true;
            int g = 0, a = 0;
            for (ItemSeq q; ok;) {
                const int w = next_item(q);
                if (w >= n_items) break;
                const Item it = item_of(w);
                if (it.n == 0) continue;
                if (a > 0) {  // K and V of the last item are free once its last S^T and dP^T are done
                    if (!(ok = bwait<PAIR>(B_KE, (a - 1) & 1, ctl, kSiteBwdQEmpty))) break;
                    if (lane == 0) {
                        load_t(it, false);
                        ++k_fills;
                    }
                    if (!(ok = bwait<PAIR>(B_VE, (a - 1) & 1, ctl, kSiteBwdQEmpty))) break;
                    if (lane == 0) {
                        load_t(it, true);
                        ++v_fills;
                    }
                } else if (!first_active && lane == 0) {
                    load_kv(it);
                    ++k_fills;
                    ++v_fills;
                }
                fetch_vec(it, it.i0);
                for (int ii = 0; ii < it.n; ++ii) {
                    const int gi = g + ii, st = gi & 1, i = it.i0 + ii;
                    if (!(ok = bwait<PAIR>(B_STE + 8 * st, ((gi >> 1) & 1) ^ 1, ctl, kSiteBwdQEmpty))) break;
                    if (lane == 0) {  // byte count first (no arrival), then the copies
                        if (lead) mbar_expect_tx(B_STF + 8 * st, (PAIR ? 4 : 2) * C::TILE);
                        if constexpr (PAIR) {
                            const uint32_t fb = lead_bar(B_STF + 8 * st);
                            const int qr = i * 128 + 64 * (int)rank, fc = 64 * (int)rank;
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const CUtensorMap* m = t ? &map_do : &map_q;
                                const uint32_t dst = t ? sDO(st) : sQ(st);
                                tma_load_3d_pair(dst, m, fb, 0, qr, it.bh, pol);                      // X0
                                tma_load_3d_pair(dst + kQuad, m, fb, 64, qr, it.bh, pol);             // X1
                                tma_load_3d_pair(dst + 2 * kQuad, m, fb, fc, i * 128, it.bh, pol);    // Y0
                                tma_load_3d_pair(dst + 3 * kQuad, m, fb, fc, i * 128 + 64, it.bh, pol);  // Y1
                            }
                        } else {
                            for (int c = 0; c < C::KCH; ++c) {
                                tma_load_3d(sQ(st) + c * C::CHUNK, &map_q, B_STF + 8 * st, c * 64, i * 128, it.bh, pol);
                                tma_load_3d(sDO(st) + c * C::CHUNK, &map_do, B_STF + 8 * st, c * 64, i * 128, it.bh, pol);
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        vec[st * 256 + lane + 32 * t] = nl2[t];
                        vec[st * 256 + 128 + lane + 32 * t] = ndl[t];
                    }
                    arrive_lead(B_STF + 8 * st);  // all 32 lanes, after their writes
                    issued |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | ((uint32_t)((gi >> 1) & 1) << st);
                    if (ii + 1 < it.n) fetch_vec(it, i + 1);
                }
                g += it.n;
                ++a;
            }
        }
        // let the loads in flight land before exit (in a pair, the even CTA's barriers
        // count the odd CTA's loads too)
        if (*abort_flag && lane == 0 && lead) {
            if (k_fills > 0) bdrain<PAIR>(B_KV, (k_fills - 1) & 1, ctl, kSiteTeardown);
            if (v_fills > 0) bdrain<PAIR>(B_VF, (v_fills - 1) & 1, ctl, kSiteTeardown);
            for (int st = 0; st < 2; ++st)
                if (issued & (1u << st))
                    bdrain<PAIR>(B_STF + 8 * st, (issued_par >> st) & 1, ctl, kSiteTeardown);
        }
    } else if (warp == C::MMA) {
        // ------------------------------------------------------------ MMA issuer 1: S^T
        // S^T(i) once S^T(i-1) has been read out of TMEM and stage i is loaded
        if (lane == 0 && lead && !*abort_flag) {
            bool ok = true;
            int g = 0, a = 0;
            for (ItemSeq q; ok;) {
                const int w = next_item(q);
                if (w >= n_items) break;
                const Item it = item_of(w);
                if (it.n == 0) continue;
                if (!(ok = bwait<PAIR>(B_KV, a & 1, ctl, kSiteBwdKvFull))) break;
                for (int ii = 0; ii < it.n; ++ii) {
                    const int gi = g + ii, st = gi & 1;
                    if (gi > 0 && !(ok = bwait<PAIR>(B_SF, (gi - 1) & 1, ctl, kSiteBwdS))) break;
                    if (!(ok = bwait<PAIR>(B_STF + 8 * st, (gi >> 1) & 1, ctl, kSiteBwdQFull))) break;
                    tc_fence_after();
                    if constexpr (PAIR)
                        issue_ss_pair<D>(tmem + C::COL_A, sK, sQ(st));
                    else
                        issue_ss<D>(tmem + C::COL_A, sK, sQ(st));
                    bcommit<PAIR>(B_S);
                    bcommit<PAIR>(B_STE + 8 * st);
                }
                if (!ok) break;
                if constexpr (!PAIR) mma_commit(B_KE);  // this item's last product that reads K
                g += it.n;
                ++a;
            }
            if (*abort_flag) {
                bcommit<PAIR>(B_TD);
                bdrain<PAIR>(B_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA2) {
        // ------------------------------------------------------------ MMA issuer 2: dP^T, dV, dK
        // dV(i) and dK(i) once P^T(i) and dS^T(i) are in TMEM; dP^T(i+1) over them (this
        // thread's products run in issue order, so it overwrites them only after both).  An
        // item's first dV and dK overwrite the accumulators once the last item's are stored.
        if (lane == 0 && lead && !*abort_flag) {
            bool ok = true;
            int g = 0, a = 0;
            for (ItemSeq q; ok;) {
                const int w = next_item(q);
                if (w >= n_items) break;
                const Item it = item_of(w);
                if (it.n == 0) continue;
                if (!(ok = bwait<PAIR>(B_VF, a & 1, ctl, kSiteBwdKvFull))) break;
                if (!(ok = bwait<PAIR>(B_STF + 8 * (g & 1), (g >> 1) & 1, ctl, kSiteBwdQFull))) break;
                tc_fence_after();
                if constexpr (PAIR)
                    issue_ss_pair<D>(tmem + C::COL_B, sV, sDO(g & 1));
                else
                    issue_ss<D>(tmem + C::COL_B, sV, sDO(g & 1));
                bcommit<PAIR>(B_DP);
                if (!PAIR && it.n == 1) mma_commit(B_VE);  // the item's last product that reads V
                for (int ii = 0; ii < it.n; ++ii) {
                    const int gi = g + ii, st = gi & 1;
                    if (!(ok = bwait<PAIR>(B_DS, gi & 1, ctl, kSiteBwdDS))) break;
                    if (ii == 0 && a > 0 && !(ok = bwait<PAIR>(B_ACCE, (a - 1) & 1, ctl, kSiteBwdDone))) break;
                    tc_fence_after();
                    if constexpr (PAIR) {
                        issue_ts_pair<D>(tmem + C::COL_ACC0, tmem + C::COL_B, sDO(st) + 2 * kQuad, ii > 0);      // dV
                        issue_ts_pair<D>(tmem + C::COL_ACC1, tmem + C::COL_B + 32, sQ(st) + 2 * kQuad, ii > 0);  // dK
                    } else {
                        issue_ts<D>(tmem + C::COL_ACC0, tmem + C::COL_B, sDO(st), ii > 0);      // dV += P^T dO
                        issue_ts<D>(tmem + C::COL_ACC1, tmem + C::COL_B + 32, sQ(st), ii > 0);  // dK += dS^T Q
                    }
                    bcommit<PAIR>(B_STE + 8 * st);
                    if (ii + 1 < it.n) {
                        if (!(ok = bwait<PAIR>(B_STF + 8 * (st ^ 1), ((gi + 1) >> 1) & 1, ctl, kSiteBwdQFull))) break;
                        tc_fence_after();
                        if constexpr (PAIR)
                            issue_ss_pair<D>(tmem + C::COL_B, sV, sDO(st ^ 1));
                        else
                            issue_ss<D>(tmem + C::COL_B, sV, sDO(st ^ 1));  // dP^T of the next query tile
                        bcommit<PAIR>(B_DP);
                        if (!PAIR && ii + 2 == it.n) mma_commit(B_VE);  // the item's last product that reads V
                    }
                }
                if (!ok) break;
                bcommit<PAIR>(B_ACC);
                g += it.n;
                ++a;
            }
            if (*abort_flag) {
                bcommit<PAIR>(B_TD2);
                bdrain<PAIR>(B_TD2, 0, ctl, kSiteTeardown);
            }
        }
    } else if (warp < C::PRODUCER) {
        // ------------------------------------------------------------ P^T, dS^T, epilogue
        // Two warpgroups: warpgroup h handles query columns [64h, 64h + 64) of every key row.
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // key row within the tile = TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t colA = C::COL_A + 64 * h, colB = C::COL_B + 64 * h;
        const float sc = p.scale_log2;
        // in a pair every wait is made warp-uniform (the TMEM loads that follow are warp-collective),
        // and each warp's arrival is one elected thread's, after the warp's TMEM accesses
        auto wait_c = [&](uint32_t b, uint32_t par, int site) {
            bool w = bwait<PAIR>(b, par, ctl, site);
            if constexpr (PAIR) w = __all_sync(0xffffffffu, w);
            return w;
        };
        auto arrive_c = [&](uint32_t b) {
            if constexpr (PAIR) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(b, 0));
            } else {
                mbar_arrive(b);
            }
        };
        bool ok = true;
        int g = 0, a = 0;
        for (ItemSeq q; ok;) {
            const int w = next_item(q);
            if (w >= n_items) break;
            const Item it = item_of(w);
            const int kg = it.kt * 128 + r;
            const bool row_ok = kg < p.Nk;    // stored (zeros past the sequence)
            const bool key_ok = kg < it.nk;   // a key of the sequence
            const int off = it.off;
            for (int ii = 0; ii < it.n; ++ii) {
                const int gi = g + ii, st = gi & 1, i = it.i0 + ii;
                const float* l2 = vec + st * 256 + 64 * h;
                const float* dl = l2 + 128;
                // key kg is visible to query q iff kg <= q + off, i.e. column c >= cmin
                const int cmin = p.causal ? kg - off - i * 128 - 64 * h : -1;
                if (!(ok = wait_c(B_S, gi & 1, kSiteBwdS))) break;
                tc_fence_after();
                uint32_t pp[32];
                uint32_t va[32], vb[32];
                // read this warpgroup's 64 S^T columns, then release them: the next S^T may overwrite
                tmem_ld32_async(lane_addr + colA, va);
                tmem_ld32_async(lane_addr + colA + 32, vb);
                tmem_wait_ld(va);
                tmem_wait_ld(vb);
                tc_fence_before();
                arrive_c(B_SF);
                // masked entries: rows past Nk (whole row) and, causal, columns c < cmin.
                // Tiles with none in the warp take the instantiation without the test.
                const int cmin_eff = key_ok ? cmin : (1 << 30);
                // sliding window: queries c > cmax_w no longer see key kg
                const int cmax_w = p.window > 0 ? kg - off + p.window - 1 - i * 128 - 64 * h : (1 << 30);
                auto p_phase = [&](auto MASK) {
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint32_t(&v)[32] = q4 ? vb : va;
                    float lv[32];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 t = reinterpret_cast<const float4*>(l2 + q4 * 32)[e];
                        lv[4 * e] = t.x, lv[4 * e + 1] = t.y, lv[4 * e + 2] = t.z, lv[4 * e + 3] = t.w;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c0 = q4 * 32 + 2 * e;
                        const float2 x = ffma2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                               make_float2(sc, sc), make_float2(-lv[2 * e], -lv[2 * e + 1]));
                        float pa = ex2(x.x), pb = ex2(x.y);
                        if constexpr (decltype(MASK)::value) {
                            if (c0 < cmin_eff || c0 > cmax_w) pa = 0.f;
                            if (c0 + 1 < cmin_eff || c0 + 1 > cmax_w) pb = 0.f;
                        }
                        pp[q4 * 16 + e] = pack_bf16(pa, pb);
                    }
                }
                };
                if (__any_sync(0xffffffffu, cmin_eff > 0 || cmax_w < 63))
                    p_phase(std::true_type{});
                else
                    p_phase(std::false_type{});
                if (!(ok = wait_c(B_DP, gi & 1, kSiteBwdDP))) break;
                tc_fence_after();
                // this warpgroup's 64 dP^T columns; once both chunks are in registers, its bf16 P^T
                // goes over the first 32 of them and dS^T over the last 32
                tmem_ld32_async(lane_addr + colB, va);
                tmem_ld32_async(lane_addr + colB + 32, vb);
                tmem_wait_ld(va);
                tmem_wait_ld(vb);
                tmem_st32_async(lane_addr + colB, pp);
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint32_t(&v)[32] = q4 ? vb : va;
                    float dv[32];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 t = reinterpret_cast<const float4*>(dl + q4 * 32)[e];
                        dv[4 * e] = t.x, dv[4 * e + 1] = t.y, dv[4 * e + 2] = t.z, dv[4 * e + 3] = t.w;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t pr = pp[q4 * 16 + e];
                        const float da = bf_lo(pr) * (__uint_as_float(v[2 * e]) - dv[2 * e]);
                        const float db = bf_hi(pr) * (__uint_as_float(v[2 * e + 1]) - dv[2 * e + 1]);
                        pk[e] = pack_bf16(da, db);
                    }
                    tmem_st16_async(lane_addr + colB + 32 + q4 * 16, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                arrive_c(B_DS);
            }
            if (!ok) break;
            const bool have = it.n > 0;
            if (have) {
                if (!(ok = wait_c(B_ACC, a & 1, kSiteBwdDone))) break;
                tc_fence_after();
            }
            const size_t base = ((size_t)it.bh * p.Nk + (row_ok ? kg : 0)) * D;
            store_acc_row<D>(lane_addr + C::COL_ACC0, p.dv + base, 1.f, row_ok, !have, h * (D / 2));
            store_acc_row<D>(lane_addr + C::COL_ACC1, p.dk + base, p.scale, row_ok, !have, h * (D / 2));
            if (have) {
                if constexpr (!PAIR) {  // the accumulators are read out: the next item may overwrite them
                    tc_fence_before();
                    mbar_arrive(B_ACCE);
                }
                g += it.n;
                ++a;
            }
        }
    }
    if constexpr (PAIR) {  // a CTA that gave up stops its partner's waits too
        if (tid == 0 && *abort_flag) st_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u), 1u);
    }
    bwd_teardown<D, PAIR>(tmem);
}

// ------------------------------------------------------------------ dQ (Q-tile parallel)
template <int D>
__global__ void __launch_bounds__(Bwd<D>::THREADS_DQ, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
              const BwdParams p) {
    using C = Bwd<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;  // 1024-aligned (checked in bwd_setup)
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    // QA: Q_i and dO_i written to TMEM by the compute threads; K/V ring of NST stages
    constexpr int NST = 3;
    const uint32_t B_QA = bar0, B_STF = bar0 + 8, B_STE = bar0 + 32, B_S = bar0 + 56, B_SF = bar0 + 64,
                   B_DP = bar0 + 72, B_DS = bar0 + 80, B_ACC = bar0 + 88, B_TD = bar0 + 96;
    const uint32_t counts[13] = {256, 1, 1, 1, 1, 1, 1, 1, 256, 1, 256, 1, 1};
    // TMEM: S at 0, dP at 128 (dS bf16 over it), dQ at 256, Q_i at 384, dO_i after it (bf16 pairs)
    constexpr uint32_t COL_QA = 384, COL_DOA = 384 + D / 2;
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const uint32_t tmem = bwd_setup<D>(smem, bar0, ctl, counts, 13);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Work items: query tiles in the chunked order (causal: late query tiles, the most keys,
    // first; heads in L2-sized chunks), taken persistently as the dK/dV pass takes its key tiles.
    // The K/V ring runs on across items, so the next item's first key tiles load while this one
    // finishes.
    const int n_items = p.n_qt * p.BH;
    const int chunk_items = p.hc_q * p.n_qt;
    struct Item {
        int bh, it, nq, nk, off, n, jlo;  // n key tiles from jlo
    };
    auto item_of = [&](int w) {
        Item t;
        int mr;
        chunked_order(w, p.n_qt, p.BH, p.hc_q, t.bh, mr);
        t.it = p.causal ? p.n_qt - 1 - mr : mr;  // causal: late query tiles (most keys) first
        bwd_seqlen(p, t.bh, t.nq, t.nk);
        t.off = t.nk - t.nq;
        int n = t.it * 128 < t.nq ? (t.nk + 127) / 128 : 0;  // a tile wholly past the sequence only stores zeros
        if (p.causal && n > 0) {
            const int qmax = min(t.it * 128 + 127, t.nq - 1);
            const long long lim = (long long)qmax + t.off;
            n = lim < 0 ? 0 : min(n, (int)(lim / 128) + 1);
        }
        int jlo = 0;  // sliding window: first key tile the tile's first query sees
        if (p.window > 0) {
            const long long lo = (long long)t.it * 128 + t.off - p.window + 1;
            jlo = lo <= 0 ? 0 : (int)min((long long)n, lo / 128);
        }
        t.jlo = jlo;
        t.n = n - jlo;
        return t;
    };
    static_assert(NST * 2 * C::TILE <= C::OFF_VEC, "K/V stages fit below the vector region");
    auto sK = [&](int st) { return s_base + st * 2 * C::TILE; };
    auto sV = [&](int st) { return s_base + st * 2 * C::TILE + C::TILE; };

    // Every role counts the key tiles (g) and the items with at least one (a) it has taken: the
    // ring and the per-tile barriers follow g, B_QA and B_ACC follow a.
    if (warp == C::PRODUCER) {
        if (lane == 0 && !*abort_flag) {
            const uint64_t pol = l2_policy_evict_last();
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            uint32_t issued = 0, issued_par = 0;
            bool ok = true;
            int g = 0;
            for (ItemSeq q; ok;) {
                const int w = next_chunked_item(q, n_items, chunk_items, gridDim.x, blockIdx.x, p.causal != 0);
                if (w >= n_items) break;
                const Item t = item_of(w);
                for (int jj = 0; jj < t.n; ++jj) {
                    const int gj = g + jj, st = gj % NST;
                    const uint32_t ph = (uint32_t)((gj / NST) & 1);
                    if (!(ok = mbar_wait(B_STE + 8 * st, ph ^ 1, ctl, kSiteBwdQEmpty))) break;
                    mbar_arrive_expect_tx(B_STF + 8 * st, 2 * C::TILE);
                    for (int c = 0; c < C::KCH; ++c) {
                        tma_load_3d(sK(st) + c * C::CHUNK, &map_k, B_STF + 8 * st, c * 64, (t.jlo + jj) * 128, t.bh, pol);
                        tma_load_3d(sV(st) + c * C::CHUNK, &map_v, B_STF + 8 * st, c * 64, (t.jlo + jj) * 128, t.bh, pol);
                    }
                    issued |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (ph << st);
                }
                g += t.n;
            }
            if (*abort_flag) {
                for (int st = 0; st < NST; ++st)
                    if (issued & (1u << st)) mbar_drain(B_STF + 8 * st, (issued_par >> st) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0 && !*abort_flag) {
            bool ok = true;
            int g = 0, a = 0;
            for (ItemSeq q; ok;) {
                const int w = next_chunked_item(q, n_items, chunk_items, gridDim.x, blockIdx.x, p.causal != 0);
                if (w >= n_items) break;
                const Item t = item_of(w);
                if (t.n == 0) continue;
                // Q and dO of this item in TMEM; written after every product of the last item
                // (which read them, and its dQ) is done and its dQ has been read out
                if (!(ok = mbar_wait(B_QA, a & 1, ctl, kSiteBwdQFull))) break;
                if (!(ok = mbar_wait(B_STF + 8 * (g % NST), (g / NST) & 1, ctl, kSiteBwdKvFull))) break;
                tc_fence_after();
                issue_ts_k<D>(tmem + C::COL_A, tmem + COL_QA, sK(g % NST));   // S = Q K^T, Q from TMEM
                mma_commit(B_S);
                issue_ts_k<D>(tmem + C::COL_B, tmem + COL_DOA, sV(g % NST));  // dP = dO V^T, dO from TMEM
                mma_commit(B_DP);
                for (int jj = 0; jj < t.n; ++jj) {
                    const int gj = g + jj, st = gj % NST, stn = (gj + 1) % NST;
                    const bool more = jj + 1 < t.n;
                    if (more) {
                        if (!(ok = mbar_wait(B_SF, gj & 1, ctl, kSiteBwdP))) break;
                        if (!(ok = mbar_wait(B_STF + 8 * stn, ((gj + 1) / NST) & 1, ctl, kSiteBwdKvFull))) break;
                        tc_fence_after();
                        issue_ts_k<D>(tmem + C::COL_A, tmem + COL_QA, sK(stn));
                        mma_commit(B_S);
                    }
                    if (!(ok = mbar_wait(B_DS, gj & 1, ctl, kSiteBwdDS))) break;
                    tc_fence_after();
                    issue_ts<D>(tmem + C::COL_ACC0, tmem + C::COL_B, sK(st), jj > 0);  // dQ += dS K
                    mma_commit(B_STE + 8 * st);
                    if (more) {
                        issue_ts_k<D>(tmem + C::COL_B, tmem + COL_DOA, sV(stn));
                        mma_commit(B_DP);
                    }
                }
                if (!ok) break;
                mma_commit(B_ACC);
                g += t.n;
                ++a;
            }
            if (*abort_flag) {
                mma_commit(B_TD);
                mbar_drain(B_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // Two warpgroups: warpgroup h handles key columns [64h, 64h + 64) of every query row.
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // query row within the tile = TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t colA = C::COL_A + 64 * h, colB = C::COL_B + 64 * h;
        const float sc = p.scale_log2;
        bool ok = true;
        int g = 0, a = 0;
        for (ItemSeq q; ok;) {
            const int w = next_chunked_item(q, n_items, chunk_items, gridDim.x, blockIdx.x, p.causal != 0);
            if (w >= n_items) break;
            const Item t = item_of(w);
            const int n = t.n, jlo = t.jlo, off = t.off, bh = t.bh;
            const int qg = t.it * 128 + r;
            const bool row_ok = qg < p.Nq;
            float l2 = INFINITY, dl = 0.f;
            if (qg < t.nq) {  // a row past the sequence keeps P = 0
                const float L = p.lse[(size_t)bh * p.Nq + qg];
                l2 = (L == -INFINITY) ? INFINITY : L * kLog2e;
                dl = p.delta[(size_t)bh * p.Nq + qg];
            }
            const int lim_row = p.causal ? min(qg + off, t.nk - 1) : t.nk - 1;  // last key this row sees
            // Q_i and dO_i into TMEM as the A operands of the score products: row = lane,
            // bf16 pairs in column order; warpgroup h writes d-columns [h D/2, (h+1) D/2)
            if (n > 0) {
                // both half rows' loads in flight before the first TMEM store (32-byte loads
                // where the rows allow: a warp instruction touches each row's line once per 32 bytes)
                constexpr int NC = D / 64;  // 64-byte pieces per half row (D / 2 bf16)
                const size_t ro = ((size_t)bh * p.Nq + (row_ok ? qg : 0)) * D + h * (D / 2);
                const bool wide = (((uintptr_t)(p.q + ro) | (uintptr_t)(p.dO + ro)) & 31) == 0;
                uint32_t wq[NC][16], wo[NC][16];
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    if (row_ok) {
                        load_row64_nc(p.q + ro + 32 * c, wq[c], wide);
                        load_row64_nc(p.dO + ro + 32 * c, wo[c], wide);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) wq[c][i] = wo[c][i] = 0u;
                    }
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    tmem_st16_async(lane_addr + COL_QA + h * (D / 4) + 16 * c, wq[c]);
                    tmem_st16_async(lane_addr + COL_DOA + h * (D / 4) + 16 * c, wo[c]);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(B_QA);
            }
            for (int jj = 0; jj < n; ++jj) {
                const int gj = g + jj;
                const int kb = (jlo + jj) * 128 + 64 * h;           // key of this warpgroup's column 0
                const int cmax = lim_row - kb;                       // columns > cmax are masked
                const int cmin_w = p.window > 0 ? qg + off - p.window + 1 - kb : -(1 << 30);  // and < cmin_w
                if (jj + 1 == n) {  // the next item's Q and dO rows towards L2 while this one finishes
                    ItemSeq qn = q;
                    const int wn = next_chunked_item(qn, n_items, chunk_items, gridDim.x, blockIdx.x, p.causal != 0);
                    if (wn < n_items) {
                        int bhn, mrn;
                        chunked_order(wn, p.n_qt, p.BH, p.hc_q, bhn, mrn);
                        const int qn_row = (p.causal ? p.n_qt - 1 - mrn : mrn) * 128 + r;
                        if (qn_row < p.Nq) {
                            const size_t o = ((size_t)bhn * p.Nq + qn_row) * D + h * (D / 2);
                            asm volatile("prefetch.L2 [%0];" ::"l"(p.q + o));
                            asm volatile("prefetch.L2 [%0];" ::"l"(p.dO + o));
                        }
                    }
                }
                if (!(ok = mbar_wait(B_S, gj & 1, ctl, kSiteBwdS))) break;
                tc_fence_after();
                uint32_t pp[32];
                uint32_t va[32], vb[32];
                // read this warpgroup's 64 S columns, then release them: the next S may overwrite
                tmem_ld32_async(lane_addr + colA, va);
                tmem_ld32_async(lane_addr + colA + 32, vb);
                tmem_wait_ld(va);
                tmem_wait_ld(vb);
                tc_fence_before();
                mbar_arrive(B_SF);
                // masked entries: columns c > cmax (keys past Nk or, causal, past the
                // row's limit); tiles with none in the warp skip the test.
                auto p_phase = [&](auto MASK) {
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint32_t(&v)[32] = q4 ? vb : va;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c0 = q4 * 32 + 2 * e;
                        const float2 x = ffma2(make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])),
                                               make_float2(sc, sc), make_float2(-l2, -l2));
                        float pa = ex2(x.x), pb = ex2(x.y);
                        if constexpr (decltype(MASK)::value) {
                            if (c0 > cmax || c0 < cmin_w) pa = 0.f;
                            if (c0 + 1 > cmax || c0 + 1 < cmin_w) pb = 0.f;
                        }
                        pp[q4 * 16 + e] = pack_bf16(pa, pb);
                    }
                }
                };
                if (__any_sync(0xffffffffu, cmax < 63 || cmin_w > 0))
                    p_phase(std::true_type{});
                else
                    p_phase(std::false_type{});
                if (!(ok = mbar_wait(B_DP, gj & 1, ctl, kSiteBwdDP))) break;
                tc_fence_after();
                tmem_ld32_async(lane_addr + colB, va);
                tmem_wait_ld(va);
                tmem_ld32_async(lane_addr + colB + 32, vb);
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                    uint32_t(&v)[32] = q4 ? vb : va;
                    if (q4) tmem_wait_ld(vb);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t pr = pp[q4 * 16 + e];
                        pk[e] = pack_bf16(bf_lo(pr) * (__uint_as_float(v[2 * e]) - dl),
                                          bf_hi(pr) * (__uint_as_float(v[2 * e + 1]) - dl));
                    }
                    tmem_st16_async(lane_addr + colB + q4 * 16, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(B_DS);
            }
            if (!ok) break;
            const bool have = n > 0;
            if (have) {
                if (!(ok = mbar_wait(B_ACC, a & 1, ctl, kSiteBwdDone))) break;
                tc_fence_after();
            }
            store_acc_row<D>(lane_addr + C::COL_ACC0, p.dq + ((size_t)bh * p.Nq + (row_ok ? qg : 0)) * D,
                             p.scale, row_ok, !have, h * (D / 2));
            if (have) {
                g += n;
                ++a;
            }
        }
    }
    bwd_teardown<D>(tmem);
    // When launched to overlap the end of the dK/dV grid, this grid must not finish before
    // it: work that follows both on the stream may read dK and dV once this grid is done.
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ single pass: dK, dV and dQ
// One CTA per (b, h, 128-key tile), as the dK/dV pass, over query tiles of 64
// rows, with the fifth product in the same pass: dQ_i += scale dS_ij K_j is
// computed as its transpose dQ^T = K^T dS^T (M = the 128 features, N = 64
// queries, K = the 128 keys), staged in shared memory as [64 queries][128
// features] fp32 and added to an fp32 accumulator in global memory by one bulk
// reduce-add (cp.reduce.async.bulk ... add.f32: the tile's rows are contiguous
// there too) per tile, so no pass recomputes S and dP for dQ.  dS^T is staged
// once in shared memory ([128 keys][64 queries] bf16, 128-byte swizzle), where
// it is both the K-major A operand of dK += dS^T Q and the MN-major B operand
// of dQ^T; K^T is the resident K tile read MN-major.  The order of the fp32
// additions into dQ varies from run to run (the result does not otherwise).
//   TMEM: S^T 64 | dP^T two buffers x 64 (P^T bf16 over each) | dQ^T 64 | dV 128 | dK 128
//   issuer 1 (warp 9): S^T(i) once S^T(i-1) has been read out.
//   issuer 2 (warp 10): dP^T(i+1) into buffer (i+1) & 1 as soon as its stage is
//     loaded (P^T(i-1) there was read by dV(i-1), issued before it: this
//     thread's products run in issue order); then dV(i), dK(i) once P^T(i),
//     dS^T(i) are written; then dQ^T(i) once the compute threads have read
//     dQ^T(i-1) out.  So the next tile's dP^T never waits for this tile's
//     dV and dK.
//   compute (warps 0-7, thread = key row; warpgroup h: query columns 32h..32h+31):
//     P phase, dS phase (P^T to TMEM, dS^T to shared memory), then the read-out
//     of dQ^T(i-1) (thread = feature row) into the staging tile, whose
//     reduce-add one of them then issues; dV, dK epilogue.
struct Fu {
    static constexpr int D = 128;
    static constexpr int BQ = 64;                    // query rows per tile
    static constexpr int NST = 3;                    // Q / dO stages
    static constexpr int KV_TILE = 128 * D * 2;      // 32 KB
    static constexpr int CHUNK = 128 * 128;          // 64 features x 128 keys
    static constexpr int QT = BQ * D * 2;            // one Q or dO tile, 16 KB
    static constexpr int QCH = BQ * 128;             // 64 features x 64 rows
    static constexpr int OFF_K = 0, OFF_V = KV_TILE;
    static constexpr int OFF_ST = 2 * KV_TILE;       // stage s: Q at + 2s QT, dO after it
    static constexpr int DS_BYTES = 128 * BQ * 2;    // dS^T [128 keys][64 queries] bf16
    static constexpr int OFF_DS = OFF_ST + NST * 2 * QT;  // two dS^T buffers
    static constexpr int OFF_DQS = OFF_DS + 2 * DS_BYTES;  // dQ staging [64 queries][128 features] fp32
    static constexpr int OFF_VEC = OFF_DQS + BQ * D * 4;   // stage s: 64 lse2 at [128 s], 64 delta after
    static constexpr int OFF_BAR = OFF_VEC + NST * 2 * BQ * 4;
    static constexpr int NBAR = 22;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16;
    static constexpr int THREADS = 352;
    static constexpr int PRODUCER = 8, MMA = 9, MMA2 = 10;
    static constexpr uint32_t COL_S = 0, COL_DP = 64, COL_DQ = 192, COL_DV = 256, COL_DK = 384;  // dP^T b at 64 + 64 b
    static constexpr uint32_t ID_S = idesc_bf16(128, BQ, 0, 0);    // S^T, dP^T: K-major A and B
    static constexpr uint32_t ID_VK = idesc_bf16(128, D, 0, 1);    // dV, dK: B (dO, Q) MN-major
    static constexpr uint32_t ID_Q = idesc_bf16(128, BQ, 1, 1);    // dQ^T: K^T and dS^T both MN-major
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(OFF_ST % 1024 == 0 && OFF_DS % 1024 == 0 && OFF_DQS % 128 == 0, "tile alignment");
};

__global__ void __launch_bounds__(Fu::THREADS, 1)
bwd_fused_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                 const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                 const BwdParams p) {
    using C = Fu;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    const uint32_t B_KV = bar0, B_STF = bar0 + 8, B_STE = bar0 + 32, B_S = bar0 + 56, B_SF = bar0 + 64,
                   B_DP = bar0 + 72, B_DS = bar0 + 88, B_DSF = bar0 + 96, B_DQ = bar0 + 112, B_QF = bar0 + 120,
                   B_ACC = bar0 + 128, B_TD = bar0 + 136, B_TD2 = bar0 + 144, B_QSF = bar0 + 152,
                   B_QSW = bar0 + 160, B_DS1 = bar0 + 168;
    // KV, STF[3] (producer lanes), STE[3] (both issuers), S, SF (compute threads), DP[2], DS[2]
    // (compute: DS for even tiles, DS1 for odd ones), DSF[2], DQ, QF (compute), ACC, TD, TD2, QSF
    // (dQ staging free: thread 0), QSW (dQ staging written: compute threads).  DS alternates:
    // dP^T(i+1) is issued before dS(i) is waited for, so a warp can form dS(i+1) while another still
    // forms dS(i), and one barrier would count both tiles' arrivals in one phase; tile i+2 needs
    // dQ^T(i), hence every arrival for tile i, so two barriers never mix.
    const uint32_t counts[C::NBAR] = {1, 32, 32, 32, 2, 2, 2, 1, 256, 1, 1, 256, 1, 1, 1, 256, 1, 1, 1, 1, 256, 256};
    uint32_t* tmem_slot = (uint32_t*)(smem + C::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        *abort_flag = 0;
        for (int b = 0; b < C::NBAR; ++b) mbar_init(bar0 + 8 * b, counts[b]);
        fence_mbar_init();
        if ((s_base & 1023u) != 0) record_error(ctl, kErrTimeout, kSiteAlign, 0);
    }
    if (warp == C::MMA) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int bh, kt;  // key tile 0 (the most query tiles when causal) first, heads in L2-sized chunks
    chunked_order(blockIdx.x, p.n_kt, p.BH, p.hc_fu, bh, kt);
    int nq, nk;
    bwd_seqlen(p, bh, nq, nk);
    const int off = nk - nq;
    int i0 = 0;
    if (p.causal) {
        const int first_q = kt * 128 - off;  // smallest query that sees key kt*128
        i0 = first_q <= 0 ? 0 : first_q / C::BQ;
    }
    int i_end = kt * 128 < nk ? (nq + C::BQ - 1) / C::BQ : 0;
    if (p.window > 0) {
        const long long qlast = (long long)kt * 128 + 127 - off + p.window - 1;
        i_end = qlast < 0 ? 0 : (int)min((long long)i_end, qlast / C::BQ + 1);
    }
    const int n = i0 < i_end ? i_end - i0 : 0;
    const uint32_t sK = s_base + C::OFF_K, sV = s_base + C::OFF_V;
    auto sQ = [&](int st) { return s_base + C::OFF_ST + st * 2 * C::QT; };
    auto sDO = [&](int st) { return s_base + C::OFF_ST + st * 2 * C::QT + C::QT; };
    auto sDS = [&](int b) { return s_base + C::OFF_DS + b * C::DS_BYTES; };
    float* vec = (float*)(smem + C::OFF_VEC);
    const bool kv_issued = warp == C::PRODUCER && lane == 0 && n > 0 && !*abort_flag;
    if (kv_issued) {  // K and V do not come from the preprocess: they load before the wait for it
        mbar_arrive_expect_tx(B_KV, 2 * C::KV_TILE);
        for (int c = 0; c < 2; ++c) {
            tma_load_3d(sK + c * C::CHUNK, &map_k, B_KV, c * 64, kt * 128, bh, l2_policy_evict_last());
            tma_load_3d(sV + c * C::CHUNK, &map_v, B_KV, c * 64, kt * 128, bh, l2_policy_evict_last());
        }
    }
    // D and the zeroed dQ accumulator come from the preprocess
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == C::PRODUCER) {
        // ------------------------------------------------------------ producer (whole warp)
        if (!*abort_flag && n > 0) {
            const uint64_t pol = l2_policy_evict_last();
            if (lane == 0) {
                tma_prefetch_desc(&map_q);
                tma_prefetch_desc(&map_do);
            }
            uint32_t issued = 0, issued_par = 0;
            float nl2[2], ndl[2];
            auto fetch_vec = [&](int i) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int q = i * C::BQ + lane + 32 * t;
                    nl2[t] = INFINITY;
                    ndl[t] = 0.f;
                    if (q < nq) {
                        const float L = p.lse[(size_t)bh * p.Nq + q];
                        nl2[t] = (L == -INFINITY) ? INFINITY : L * kLog2e;
                        ndl[t] = p.delta[(size_t)bh * p.Nq + q];
                    }
                }
            };
            fetch_vec(i0);
            for (int ii = 0; ii < n; ++ii) {
                const int st = ii % C::NST, i = i0 + ii;
                const uint32_t use = (uint32_t)(ii / C::NST);
                if (!mbar_wait(B_STE + 8 * st, (use & 1) ^ 1, ctl, kSiteBwdQEmpty)) break;
                if (lane == 0) {
                    mbar_expect_tx(B_STF + 8 * st, 2 * C::QT);
                    for (int c = 0; c < 2; ++c) {
                        tma_load_3d(sQ(st) + c * C::QCH, &map_q, B_STF + 8 * st, c * 64, i * C::BQ, bh, pol);
                        tma_load_3d(sDO(st) + c * C::QCH, &map_do, B_STF + 8 * st, c * 64, i * C::BQ, bh, pol);
                    }
                }
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    vec[st * 128 + lane + 32 * t] = nl2[t];
                    vec[st * 128 + 64 + lane + 32 * t] = ndl[t];
                }
                mbar_arrive(B_STF + 8 * st);
                issued |= 1u << st;
                issued_par = (issued_par & ~(1u << st)) | ((use & 1) << st);
                if (ii + 1 < n) fetch_vec(i + 1);
            }
            if (*abort_flag && lane == 0) {
                if (kv_issued) mbar_drain(B_KV, 0, ctl, kSiteTeardown);
                for (int st = 0; st < C::NST; ++st)
                    if (issued & (1u << st)) mbar_drain(B_STF + 8 * st, (issued_par >> st) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA) {
        // ------------------------------------------------------------ issuer 1: S^T
        if (lane == 0 && !*abort_flag && n > 0) {
            bool ok = mbar_wait(B_KV, 0, ctl, kSiteBwdKvFull);
            for (int ii = 0; ii < n && ok; ++ii) {
                const int st = ii % C::NST;
                if (ii >= 1 && !(ok = mbar_wait(B_SF, (ii - 1) & 1, ctl, kSiteBwdS))) break;
                if (!(ok = mbar_wait(B_STF + 8 * st, (ii / C::NST) & 1, ctl, kSiteBwdQFull))) break;
                tc_fence_after();
                const uint64_t a0 = sdesc_sw128(sK, 16, 1024), b0 = sdesc_sw128(sQ(st), 16, 1024);
                const uint32_t d = tmem + C::COL_S;
                mma_ss_first(d, a0, b0, C::ID_S);
#pragma unroll
                for (int k = 1; k < 8; ++k)
                    mma_ss_acc(d, sdesc_add(a0, (k >> 2) * C::CHUNK + (k & 3) * 32),
                               sdesc_add(b0, (k >> 2) * C::QCH + (k & 3) * 32), C::ID_S);
                mma_commit(B_S);
                mma_commit(B_STE + 8 * st);
            }
            if (*abort_flag) {
                mma_commit(B_TD);
                mbar_drain(B_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA2) {
        // ------------------------------------------------------------ issuer 2: dP^T, dV, dK, dQ^T
        if (lane == 0 && !*abort_flag && n > 0) {
            auto issue_dp = [&](int jj) {  // dP^T of tile jj into buffer jj & 1, once its stage is loaded
                const int st = jj % C::NST;
                if (!mbar_wait(B_STF + 8 * st, (jj / C::NST) & 1, ctl, kSiteBwdQFull)) return false;
                tc_fence_after();
                const uint64_t a0 = sdesc_sw128(sV, 16, 1024), b0 = sdesc_sw128(sDO(st), 16, 1024);
                const uint32_t d = tmem + C::COL_DP + 64 * (jj & 1);
                mma_ss_first(d, a0, b0, C::ID_S);
#pragma unroll
                for (int k = 1; k < 8; ++k)
                    mma_ss_acc(d, sdesc_add(a0, (k >> 2) * C::CHUNK + (k & 3) * 32),
                               sdesc_add(b0, (k >> 2) * C::QCH + (k & 3) * 32), C::ID_S);
                mma_commit(B_DP + 8 * (jj & 1));
                return true;
            };
            bool ok = mbar_wait(B_KV, 0, ctl, kSiteBwdKvFull);
            if (ok) ok = issue_dp(0);
            for (int ii = 0; ii < n && ok; ++ii) {
                const int st = ii % C::NST, b = ii & 1;
                if (ii + 1 < n && !(ok = issue_dp(ii + 1))) break;
                if (!(ok = mbar_wait((ii & 1) ? B_DS1 : B_DS, (ii >> 1) & 1, ctl, kSiteBwdDS))) break;
                tc_fence_after();
                const bool acc = ii > 0;
                {   // dV += P^T dO: A = P^T (TMEM; k-step k = queries 16k.., warpgroup k / 2's
                    // columns), B = dO MN-major (64-feature blocks 8 KB apart, 16 rows per k-step)
                    const uint64_t bv = sdesc_sw128(sDO(st), C::QCH, 1024);
                    const uint64_t bq = sdesc_sw128(sQ(st), C::QCH, 1024);
                    const uint64_t ad = sdesc_sw128(sDS(b), 16, 1024);  // dS^T K-major: 16 queries per k-step
                    const uint32_t pcol = tmem + C::COL_DP + 64 * b;
                    mma_ts(tmem + C::COL_DV, pcol, bv, C::ID_VK, acc ? 1u : 0u);
#pragma unroll
                    for (int k = 1; k < 4; ++k)
                        mma_ts_acc(tmem + C::COL_DV, pcol + 32 * (k >> 1) + 8 * (k & 1), sdesc_add(bv, k * 2048),
                                   C::ID_VK);
                    // dK += dS^T Q: A = dS^T from shared memory (K-major), B = Q MN-major
                    mma_ss(tmem + C::COL_DK, ad, bq, C::ID_VK, acc ? 1u : 0u);
#pragma unroll
                    for (int k = 1; k < 4; ++k)
                        mma_ss_acc(tmem + C::COL_DK, sdesc_add(ad, k * 32), sdesc_add(bq, k * 2048), C::ID_VK);
                }
                mma_commit(B_STE + 8 * st);
                // dQ^T(ii) = K^T dS^T once dQ^T(ii-1) has been read out: A = K MN-major (feature
                // blocks 16 KB apart, 16 keys per k-step), B = dS^T MN-major (16 keys per k-step)
                if (ii > 0 && !(ok = mbar_wait(B_QF, (ii - 1) & 1, ctl, kSiteBwdDQ))) break;
                tc_fence_after();
                {
                    const uint64_t ak = sdesc_sw128(sK, C::CHUNK, 1024), bs = sdesc_sw128(sDS(b), 8192, 1024);
                    mma_ss_first(tmem + C::COL_DQ, ak, bs, C::ID_Q);
#pragma unroll
                    for (int k = 1; k < 8; ++k)
                        mma_ss_acc(tmem + C::COL_DQ, sdesc_add(ak, k * 2048), sdesc_add(bs, k * 2048), C::ID_Q);
                }
                mma_commit(B_DQ);
                mma_commit(B_DSF + 8 * b);
            }
            if (ok) mma_commit(B_ACC);
            if (*abort_flag) {
                mma_commit(B_TD2);
                mbar_drain(B_TD2, 0, ctl, kSiteTeardown);
            }
        }
    } else if (warp < C::PRODUCER) {
        // ------------------------------------------------------------ compute: P, dS, dQ read-out, epilogue
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // key row (TMEM lane) = feature row of dQ^T
        const int kg = kt * 128 + r;
        const bool row_ok = kg < p.Nk;
        const bool key_ok = kg < nk;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sc = p.scale_log2;
        uint8_t* ds_row = smem + C::OFF_DS + r * 128;  // row r of a dS^T buffer (+ b * DS_BYTES)
        float* dqs = reinterpret_cast<float*>(smem + C::OFF_DQS) + r;  // column r of the dQ staging tile
        auto read_dq = [&](int jj) {  // dQ^T of tile jj: this thread's feature r, queries 32h..32h+31
            bool w = mbar_wait(B_DQ, jj & 1, ctl, kSiteBwdDQ);
            if (!__all_sync(0xffffffffu, w)) return false;  // every lane votes: the TMEM load is warp-collective
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(lane_addr + C::COL_DQ + 32 * h, v);
            tc_fence_before();
            mbar_arrive(B_QF);  // dQ^T(jj + 1) may be issued over it
            // the staging tile is free once the previous reduce-add has read it (thread 0 issued
            // it and waits for its reads; every handshake here is a bounded mbarrier wait)
            if (tid == 0) {
                bulk_wait_group_read0();
                mbar_arrive(B_QSF);
            }
            w = mbar_wait(B_QSF, jj & 1, ctl, kSiteBwdDQ);
            if (!__all_sync(0xffffffffu, w)) return false;
#pragma unroll
            for (int c = 0; c < 32; ++c) dqs[(32 * h + c) * C::D] = __uint_as_float(v[c]);  // a warp: one 128-byte row
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(B_QSW);
            bool issued = true;
            if (tid == 0) {  // rows past Nq are not added (they belong to the next head); rows past a
                             // shorter sequence hold zeros (P = 0 there)
                issued = mbar_wait(B_QSW, jj & 1, ctl, kSiteBwdDQ);
                const int q0 = (i0 + jj) * C::BQ;
                const int rows = min(C::BQ, p.Nq - q0);
                if (issued && (rows <= 0 || bh >= p.BH)) {  // never: the tile range stays inside the head
                    record_error(ctl, kErrInvalid, kSiteBwdDQ, q0);
                    issued = false;
                }
                if (issued) {
                    bulk_reduce_add_f32(p.dqacc + ((size_t)bh * p.Nq + q0) * C::D, s_base + C::OFF_DQS,
                                        (uint32_t)rows * C::D * 4);
                    bulk_commit_group();
                }
            }
            return __all_sync(0xffffffffu, issued) != 0;  // the same answer in every lane of the warp
        };
        bool ok = true;
        for (int ii = 0; ii < n; ++ii) {
            const int b = ii & 1, st = ii % C::NST, i = i0 + ii;
            const float* l2 = vec + st * 128 + 32 * h;
            const float* dl = l2 + 64;
            const int cmin = p.causal ? kg - off - i * C::BQ - 32 * h : -1;  // visible iff column c >= cmin
            ok = mbar_wait(B_S, ii & 1, ctl, kSiteBwdS);
            if (!__all_sync(0xffffffffu, ok)) break;  // every lane votes: the TMEM loads are warp-collective
            tc_fence_after();
            uint32_t va[32], pp[16];
            tmem_ld32(lane_addr + C::COL_S + 32 * h, va);
            tc_fence_before();
            mbar_arrive(B_SF);
            const int cmin_eff = key_ok ? cmin : (1 << 30);
            const int cmax_w = p.window > 0 ? kg - off + p.window - 1 - i * C::BQ - 32 * h : (1 << 30);
            auto p_phase = [&](auto MASK) {
                float lv[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 t = reinterpret_cast<const float4*>(l2)[e];
                    lv[4 * e] = t.x, lv[4 * e + 1] = t.y, lv[4 * e + 2] = t.z, lv[4 * e + 3] = t.w;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c0 = 2 * e;
                    const float2 x = ffma2(make_float2(__uint_as_float(va[2 * e]), __uint_as_float(va[2 * e + 1])),
                                           make_float2(sc, sc), make_float2(-lv[2 * e], -lv[2 * e + 1]));
                    float a = ex2(x.x), bb = ex2(x.y);
                    if constexpr (decltype(MASK)::value) {
                        if (c0 < cmin_eff || c0 > cmax_w) a = 0.f;
                        if (c0 + 1 < cmin_eff || c0 + 1 > cmax_w) bb = 0.f;
                    }
                    pp[e] = pack_bf16(a, bb);
                }
            };
            if (__any_sync(0xffffffffu, cmin_eff > 0 || cmax_w < 31))
                p_phase(std::true_type{});
            else
                p_phase(std::false_type{});
            // the dS^T buffer of this tile is free once dK and dQ^T of tile ii - 2 are done
            ok = ii < 2 || mbar_wait(B_DSF + 8 * b, ((ii >> 1) & 1) ^ 1, ctl, kSiteBwdDS);
            if (ok) ok = mbar_wait(B_DP + 8 * b, (ii >> 1) & 1, ctl, kSiteBwdDP);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            tmem_ld32(lane_addr + C::COL_DP + 64 * b + 32 * h, va);
            tmem_st16_async(lane_addr + C::COL_DP + 64 * b + 32 * h, pp);  // P^T over the dP^T columns just read
            {
                float dv[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 t = reinterpret_cast<const float4*>(dl)[e];
                    dv[4 * e] = t.x, dv[4 * e + 1] = t.y, dv[4 * e + 2] = t.z, dv[4 * e + 3] = t.w;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const uint32_t pr = pp[e];
                    pk[e] = pack_bf16(bf_lo(pr) * (__uint_as_float(va[2 * e]) - dv[2 * e]),
                                      bf_hi(pr) * (__uint_as_float(va[2 * e + 1]) - dv[2 * e + 1]));
                }
                // dS^T row r, queries 32h..32h+31: 16-byte chunks 4h..4h+3, swizzled by row
                uint8_t* row = ds_row + b * C::DS_BYTES;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(row + (((4 * h + u) ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive((ii & 1) ? B_DS1 : B_DS);
            if (ii > 0 && !(ok = read_dq(ii - 1))) break;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok && n > 0) ok = read_dq(n - 1);
        if (ok) {
            const bool have = n > 0;
            if (have) {
                ok = mbar_wait(B_ACC, 0, ctl, kSiteBwdDone);
                tc_fence_after();
            }
            if (ok) {
                const size_t base = ((size_t)bh * p.Nk + (row_ok ? kg : 0)) * C::D;
                store_acc_row<128>(lane_addr + C::COL_DV, p.dv + base, 1.f, row_ok, !have, h * 64);
                store_acc_row<128>(lane_addr + C::COL_DK, p.dk + base, p.scale, row_ok, !have, h * 64);
            }
        }
    }
    if (tid == 0) bulk_wait_group0();  // the last reduce-add has landed before the grid completes
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::MMA) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// dQ = bf16(scale * dQacc): 8 elements per thread and step (two 16-byte loads,
// one 16-byte store).  Launched as a programmatic dependent of the single pass.
__global__ void __launch_bounds__(256)
bwd_dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, long long n8, float scale) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                                                     pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
    }
}

BwdParams make_params(const BwdLaunch& a) {
    BwdParams p;
    p.q = (const __nv_bfloat16*)a.q;
    p.dO = (const __nv_bfloat16*)a.dO;
    p.dq = (__nv_bfloat16*)a.dq;
    p.dk = (__nv_bfloat16*)a.dk;
    p.dv = (__nv_bfloat16*)a.dv;
    p.lse = a.lse;
    p.delta = a.delta;
    p.BH = a.B * a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.causal = a.causal;
    p.window = a.window;
    p.lens_q = a.lens_q;
    p.lens_k = a.lens_k;
    p.H = a.H;
    // heads whose streamed tiles (Q and dO for the dK/dV pass, K and V for the dQ
    // pass) fit in 64 MiB of L2 together
    const long long budget = 64ll << 20;
    const long long per_kv = 2ll * a.Nq * a.d * 2, per_q = 2ll * a.Nk * a.d * 2;
    p.hc_kv = (int)std::max(1ll, std::min((long long)p.BH, budget / per_kv));
    p.hc_q = (int)std::max(1ll, std::min((long long)p.BH, budget / per_q));
    p.n_qt = (a.Nq + 127) / 128;
    p.n_kt = (a.Nk + 127) / 128;
    p.n_pt = (p.n_kt + 1) / 2;
    const long long per_fu = (long long)a.Nq * a.d * 8;  // Q, dO bf16 and the fp32 dQ rows of a head
    p.hc_fu = (int)std::max(1ll, std::min((long long)p.BH, budget / per_fu));
    p.dqacc = a.dqacc;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.err = a.err;
    p.timeout_ns = a.timeout_ns;
    return p;
}

template <int D>
cudaError_t launch_pre_d(const BwdLaunch& a, cudaStream_t s) {
    const long long rows = (long long)a.B * a.H * a.Nq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kPreRowsPerBlock<D> - 1) / kPreRowsPerBlock<D>));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol in the kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_pre_kernel<D>, (const __nv_bfloat16*)a.o,
                                             (const __nv_bfloat16*)a.dO, a.delta, a.dqacc, rows);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// after_pre: launched right after the preprocess on the same stream, as its
// programmatic dependent (setup and the K/V loads overlap the preprocess's end).
// PAIR (d = 128): CTA pairs (clusters of two; a key tile past Nk pads an odd
// count) instead of single CTAs.
template <int D, bool PAIR>
cudaError_t launch_dkdv_d(const BwdLaunch& a, cudaStream_t s, bool after_pre) {
    using C = Bwd<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    cudaError_t e = set_smem_limit_once<bwd_dkdv_kernel<D, PAIR>>(C::SMEM);
    if (e != cudaSuccess) return e;
    const BwdParams p = make_params(a);
    cudaLaunchConfig_t cfg = {};
    // one CTA per SM at most (persistent over key tiles); a pair per key-tile pair
    const int n_items = p.n_kt * p.BH;
    cfg.gridDim = dim3((unsigned)(PAIR ? 2 * p.n_pt * p.BH : std::min(n_items, std::max(1, a.num_sms))));
    cfg.blockDim = dim3(C::THREADS_DKDV);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (PAIR) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (after_pre) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    // the pair's Q and dO maps load 64-row quadrants
    e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<D, PAIR>, PAIR ? a.map_q2 : a.map_q, a.map_k, a.map_v,
                           PAIR ? a.map_do2 : a.map_do, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// after_dkdv: launched right after the dK/dV grid on the same stream.  The two
// passes are independent (both only read the preprocess's D), so this grid is
// launched as a programmatic dependent: its CTAs may take the SMs that the
// dK/dV grid's last wave leaves free.
template <int D>
cudaError_t launch_dq_d(const BwdLaunch& a, cudaStream_t s, bool after_dkdv) {
    using C = Bwd<D>;
    cudaError_t e = set_smem_limit_once<bwd_dq_kernel<D>>(C::SMEM);
    if (e != cudaSuccess) return e;
    const BwdParams p = make_params(a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(p.n_qt * p.BH, std::max(1, a.num_sms)));  // persistent over query tiles
    cfg.blockDim = dim3(C::THREADS_DQ);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_dkdv ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D>, a.map_q, a.map_k, a.map_v, a.map_do, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The single pass after the preprocess (programmatic dependent), then the dQ
// conversion after it.  d = 128.
cudaError_t launch_fused_d(const BwdLaunch& a, cudaStream_t s) {
    cudaError_t e = set_smem_limit_once<bwd_fused_kernel>(Fu::SMEM);
    if (e != cudaSuccess) return e;
    const BwdParams p = make_params(a);
    e = launch_dependent(bwd_fused_kernel, dim3((unsigned)(p.n_kt * p.BH)), dim3(Fu::THREADS), Fu::SMEM, s,
                         a.map_q2, a.map_k, a.map_v, a.map_do2, p);
    if (e != cudaSuccess) return e;
    const long long n8 = (long long)a.B * a.H * a.Nq * a.d / 8;
    const long long blocks = std::min<long long>((n8 + 255) / 256, (long long)a.num_sms * 8);
    return launch_dependent(bwd_dq_convert_kernel, dim3((unsigned)std::max(1ll, blocks)), dim3(256), 0, s,
                            (const float*)a.dqacc, (__nv_bfloat16*)a.dq, n8, a.scale);
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_pre_d<128>(a, s) : launch_pre_d<64>(a, s);
}
cudaError_t launch_bwd_dkdv(const BwdLaunch& a, cudaStream_t s, bool after_pre) {
    return a.d == 128 ? launch_dkdv_d<128, false>(a, s, after_pre) : launch_dkdv_d<64, false>(a, s, after_pre);
}
cudaError_t launch_bwd_fused(const BwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_fused_d(a, s) : cudaErrorInvalidValue;
}
cudaError_t launch_bwd_dkdv_pair(const BwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_dkdv_d<128, true>(a, s, false) : cudaErrorInvalidValue;
}
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t s, bool after_dkdv) {
    return a.d == 128 ? launch_dq_d<128>(a, s, after_dkdv) : launch_dq_d<64>(a, s, after_dkdv);
}

}  // namespace fa
