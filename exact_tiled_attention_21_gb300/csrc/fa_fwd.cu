// Forward pass: exact attention, tiled, online softmax, one fused kernel.
//
// Method (wiki.ai-engineering.at "Flash Attention", sections "Tiling
// Algorithm" and "Lösung: Online Softmax"; johe.ru "Flash Attention: ...",
// section "Стадии вычисления", pass 1): for a block of query rows, stream the
// key/value blocks; per block compute the scores, raise the running row
// maximum, rescale what was accumulated by exp(m_old - m_new), add
// exp(S - m_new) to the running row sum and exp(S - m_new) V to the output
// accumulator; divide by the row sum at the end.  Scale, mask, softmax and the
// value product run in one kernel (zimaspace.com "Wie reduziert Flash
// Attention ...", section "Kernel-Fusion ..."), so scores never reach HBM.
//
// GB300 mapping (one persistent CTA per SM, 320 threads, 512 TMEM columns):
//   warp 8      TMA producer: Q tiles once per work tile; K_j, V_j through a
//               ring of NSLOT shared-memory slots (full/empty mbarriers).
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (fp32) and
//               O_t += P_t V_j with P_t read from TMEM, for two 128-row query
//               tiles t = 0, 1 interleaved so that the tensor core works on
//               one tile while the softmax warps work on the other.
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: thread = row
//               (TMEM lane), so row max and row sum need no shuffles.  They
//               work in the log2 domain (scores multiplied by scale*log2 e, one
//               ex2 per score), keep the running max, rescale the O
//               accumulator in TMEM only when the max grew by more than 2^8
//               (exact either way: l and O always share the same reference
//               max), write P as bf16 over the S columns, and run the
//               epilogue O / l -> bf16, LSE = (m + log2 l) ln 2.
#include <algorithm>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

template <int D>
struct Fwd {
    static constexpr int BM = 128;                // query rows per softmax tile
    static constexpr int BN = 128;                // keys per block
    static constexpr int KCH = D / 64;            // 64-element (128-byte) column chunks
    static constexpr int Q_BYTES = BM * D * 2;    // one query tile
    static constexpr int KV_BYTES = BN * D * 2;   // one K or V block
    static constexpr int CHUNK_BYTES = 128 * 128; // 128 rows x 128 bytes
    static constexpr int NSLOT = (D == 128) ? 5 : 8;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = 2 * Q_BYTES;
    static constexpr int OFF_BAR = OFF_KV + NSLOT * KV_BYTES;
    // barriers: q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], o_final[2], teardown,
    // merge_ready, merge_done (split-KV), pv_done[2] (P in its own columns), q_full/q_empty of the
    // second query buffer (split-KV tiles double-buffer their one query tile)
    static constexpr int NBAR = 2 + 2 * NSLOT + 13;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_STAGE = OFF_MISC + 16;  // split-KV: warpgroup 1's (m, l) per row
    static constexpr int SMEM = OFF_STAGE + BM * 8 + 1024;  // + alignment slack
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    // d = 64 leaves 128 TMEM columns: P_t then gets its own 64 (bf16 pairs), so S_t of the next
    // key block need not wait for P_t V_j (with 256-row tiles; split-KV tiles keep P over S)
    static constexpr bool P_OWN = D == 64;
    static constexpr uint32_t COL_P0 = 384, COL_P1 = 448;
    static constexpr uint32_t IDESC_S = idesc_bf16(128, BN, 0, 0);  // Q, K both K-major
    static constexpr uint32_t IDESC_O = idesc_bf16(128, D, 0, 1);   // P from TMEM, V MN-major
};

struct FwdParams {
    __nv_bfloat16* o;
    float* lse;
    int BH, Nq, Nk, causal;
    int window;  // > 0: causal sliding window of this many keys
    const int* lens_q;  // per-sequence query / key counts (varlen instantiation only; may be null)
    const int* lens_k;
    int H;
    int rows;  // query rows per work tile: 256 (two 128-row tiles) or 128 (split-KV)
    int n_mtiles, num_work;
    int hc;    // heads per scheduling chunk: their K and V fit in 64 MiB of L2 together
    int per_chunk;  // the CTAs take the chunks in per-chunk rounds (next_chunked_item)
    float scale_log2;
    DevError* err;
    uint64_t timeout_ns;
};

// Query and key counts of a work tile's sequence: Nq and Nk, or with
// per-sequence lengths (VL) those of its batch entry, clamped to [0, Nq] and
// [0, Nk] (bad: a length was out of range).
struct SeqLen {
    int nq, nk;
    bool bad;
};
template <bool VL>
__device__ __forceinline__ SeqLen fwd_seqlen(const FwdParams& p, int w) {
    if (!VL || w >= p.num_work) return {p.Nq, p.Nk, false};
    const int b = (w % p.BH) / p.H;
    const int lq = p.lens_q ? __ldg(p.lens_q + b) : p.Nq;
    const int lk = p.lens_k ? __ldg(p.lens_k + b) : p.Nk;
    const int nq = min(max(lq, 0), p.Nq), nk = min(max(lk, 0), p.Nk);
    return {nq, nk, nq != lq || nk != lk};
}

__device__ __forceinline__ int fwd_num_kv(const FwdParams& p, int row0, int nq, int nk) {
    if (row0 >= nq) return 0;
    const int kv_total = (nk + 127) / 128;
    if (!p.causal) return kv_total;
    const int max_row = min(row0 + p.rows - 1, nq - 1);
    const long long lim = (long long)max_row + nk - nq;  // last key the last row sees
    if (lim < 0) return 0;
    return min(kv_total, (int)(lim / 128) + 1);
}

// First key block a work tile needs: with a sliding window, the block of the
// first visible key of its first row.
template <bool WIN>
__device__ __forceinline__ int fwd_kv_first(const FwdParams& p, int row0, int nq, int nk) {
    if (!WIN || p.window <= 0) return 0;
    const long long lo = (long long)row0 + nk - nq - p.window + 1;
    return lo <= 0 ? 0 : (int)(lo / 128);
}

// Work tile w -> (bh, first row).  Heads come in chunks of hc whose K and V
// fit in L2 together, so the CTAs in flight share them there; within a chunk
// every head's row tile of one level comes before the next level (causal:
// heaviest first).  The persistent CTAs take each chunk in rounds of
// alternating direction (next_chunked_item).
__device__ __forceinline__ void fwd_decode(const FwdParams& p, int w, int& bh, int& row0) {
    const int chunk = p.hc * p.n_mtiles;
    const int c = w / chunk;
    const int r = w - c * chunk;
    const int h0 = c * p.hc;
    const int hn = min(p.hc, p.BH - h0);
    const int mr = r / hn;
    bh = h0 + (r - mr * hn);
    const int m = p.causal ? (p.n_mtiles - 1 - mr) : mr;
    row0 = m * p.rows;
}

// Pass 1 over one 128-column S row in TMEM (thread = row): the maximum of the
// raw scores.  Chunks of 32 columns are double-buffered (the next loads while
// this one is scanned).  MASKED: columns c > lim2 or c < lo2 are excluded;
// instantiated only for the blocks that hold a masked column.
template <bool MASKED>
__device__ __forceinline__ float row_max_pass(uint32_t taddr, int lim2, int lo2) {
    // eight running maxima, so that the 64 max instructions form eight short dependency chains
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
    uint32_t va[32], vb[32];
    tmem_ld32_async(taddr, va);
    tmem_wait_ld(va);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t(&v)[32] = (q4 & 1) ? vb : va;
        uint32_t(&nx)[32] = (q4 & 1) ? va : vb;
        if (q4 + 1 < 4) tmem_ld32_async(taddr + (q4 + 1) * 32, nx);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float x0 = __uint_as_float(v[i]), x1 = __uint_as_float(v[i + 1]);
            if constexpr (MASKED) {
                if (q4 * 32 + i > lim2 || q4 * 32 + i < lo2) x0 = -INFINITY;
                if (q4 * 32 + i + 1 > lim2 || q4 * 32 + i + 1 < lo2) x1 = -INFINITY;
            }
            mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x0, x1);
        }
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
}

// Pass 2: p = 2^(s c - m) for the 128 columns, their sum, and bf16 P written
// to paddr: either over the S columns already read (paddr = taddr: keys
// [32 q, 32 q + 32) to columns [16 q, 16 q + 16); the load in flight is always
// of columns >= 32 (q + 1)), or to columns of its own.
template <bool MASKED>
__device__ __forceinline__ float exp_pass(uint32_t taddr, uint32_t paddr, int lim2, int lo2, float c, float msub) {
    float2 rs[4];  // four partial sums (short dependency chains), added at the end
#pragma unroll
    for (int k = 0; k < 4; ++k) rs[k] = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(c, c), nm2 = make_float2(-msub, -msub);
    uint32_t va[32], vb[32];
    tmem_ld32_async(taddr, va);
    tmem_wait_ld(va);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t(&v)[32] = (q4 & 1) ? vb : va;
        uint32_t(&nx)[32] = (q4 & 1) ? va : vb;
        if (q4 + 1 < 4) tmem_ld32_async(taddr + (q4 + 1) * 32, nx);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float s0 = __uint_as_float(v[2 * i]), s1 = __uint_as_float(v[2 * i + 1]);
            if constexpr (MASKED) {
                if (q4 * 32 + 2 * i > lim2 || q4 * 32 + 2 * i < lo2) s0 = -INFINITY;
                if (q4 * 32 + 2 * i + 1 > lim2 || q4 * 32 + 2 * i + 1 < lo2) s1 = -INFINITY;
            }
            const float2 x = ffma2(make_float2(s0, s1), c2, nm2);  // s*c - m, two lanes
            const float2 e = make_float2(ex2(x.x), ex2(x.y));
            rs[i & 3] = fadd2(rs[i & 3], e);
            pk[i] = pack_bf16(e.x, e.y);
        }
        tmem_st16_async(paddr + q4 * 16, pk);
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    tmem_wait_st();
    const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
    return (r01.x + r23.x) + (r01.y + r23.y);
}

// WIN: the sliding-window variant; VL: per-sequence lengths (rows past a
// sequence's length give O = 0, LSE = -inf; keys past it are masked).  SPLIT:
// for grids with few work tiles, a work tile is one 128-row query tile whose
// key blocks alternate between the two softmax warpgroups (even blocks to 0,
// odd to 1), each with its own running max, sum and O in TMEM; warpgroup 0
// merges the two at the end (the LSE-weighted combine of the online
// recurrence).  Each is a separate instantiation, so the plain path carries
// none of their bounds.
template <int D, bool WIN, bool VL, bool SPLIT>
__global__ void __launch_bounds__(Fwd<D>::THREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const FwdParams p) {
    using C = Fwd<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    const uint32_t BAR_QF = bar0, BAR_QE = bar0 + 8;
    auto bar_kvf = [&](int s) { return bar0 + 16 + 8 * s; };
    auto bar_kve = [&](int s) { return bar0 + 16 + 8 * C::NSLOT + 8 * s; };
    const uint32_t BAR_S = bar0 + 16 + 16 * C::NSLOT;  // s_full[t] = BAR_S + 8t
    const uint32_t BAR_P = BAR_S + 16;                 // p_full[t]
    const uint32_t BAR_O = BAR_P + 16;                 // o_final[t]
    const uint32_t BAR_TD = BAR_O + 16;                // teardown
    const uint32_t BAR_MR = BAR_TD + 8;                // split-KV: warpgroup 1's (m, l) staged
    const uint32_t BAR_MD = BAR_MR + 8;                // split-KV: warpgroup 0 done with O_1 and (m, l)
    const uint32_t BAR_PV = BAR_MD + 8;                // pv_done[t]: P_t V_j done (P in its own columns)
    const uint32_t BAR_QF1 = BAR_PV + 16, BAR_QE1 = BAR_PV + 24;  // split-KV: second query buffer
    constexpr bool P_OWN = C::P_OWN && !SPLIT;
    uint32_t* tmem_slot = (uint32_t*)(smem + C::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's work tiles (every role walks the same sequence)
    auto next_work = [&](ItemSeq& q) {
        return next_chunked_item(q, p.num_work, p.hc * p.n_mtiles, gridDim.x, blockIdx.x, p.per_chunk != 0);
    };

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(BAR_QF, 1);
        mbar_init(BAR_QE, 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(bar_kvf(s), 1);
            mbar_init(bar_kve(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR_S + 8 * t, 1);
            mbar_init(BAR_P + 8 * t, 128);
            mbar_init(BAR_O + 8 * t, 1);
        }
        mbar_init(BAR_TD, 1);
        mbar_init(BAR_MR, 128);
        mbar_init(BAR_MD, 128);
        mbar_init(BAR_PV, 1);
        mbar_init(BAR_PV + 8, 1);
        mbar_init(BAR_QF1, 1);
        mbar_init(BAR_QE1, 1);
        fence_mbar_init();
        if ((s_base & 1023u) != 0) record_error(ctl, kErrTimeout, kSiteAlign, (int)(s_base & 1023u));
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the kernel before it on the stream, this grid may
    // start while that one finishes: the setup above overlaps its end, and every thread waits for
    // it to complete (griddepcontrol.wait) before touching global memory.  A kernel launched after
    // this one the same way may likewise start its setup on SMs this grid leaves.
    pdl_launch_dependents();

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            if (VL) pdl_wait();  // the sequence lengths
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int slot = 0;
            uint32_t phase = 0, q_iter = 0;
            uint32_t issued = 0, issued_par = 0;  // per slot: filled at least once / its last parity
            bool ok = true;
            ItemSeq seq;
            int w_next = next_work(seq);
            SeqLen sl_next = fwd_seqlen<VL>(p, w_next);
            for (int w = w_next; w < p.num_work && ok; w = w_next) {
                w_next = next_work(seq);
                const SeqLen sl = sl_next;  // loaded one tile ahead
                sl_next = fwd_seqlen<VL>(p, w_next);
                int bh, row0;
                fwd_decode(p, w, bh, row0);
                const int jlo = fwd_kv_first<WIN>(p, row0, sl.nq, sl.nk);
                const int n = max(0, fwd_num_kv(p, row0, sl.nq, sl.nk) - jlo);
                if (n == 0) continue;
                if (!VL && q_iter == 0) pdl_wait();
                // split-KV tiles alternate between the two query buffers, so the next tile's Q
                // loads while this one runs; a 256-row tile takes both
                const int qb = SPLIT ? (int)(q_iter & 1) : 0;
                const uint32_t qn = SPLIT ? (q_iter >> 1) : q_iter;  // earlier fills of buffer qb
                const uint32_t qf = qb ? BAR_QF1 : BAR_QF, qe = qb ? BAR_QE1 : BAR_QE;
                if (qn > 0 && !mbar_wait(qe, (qn - 1) & 1, ctl, kSiteQEmpty)) break;
                mbar_arrive_expect_tx(qf, (SPLIT ? 1 : 2) * C::Q_BYTES);
                for (int t = 0; t < (SPLIT ? 1 : 2); ++t)
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_3d(s_base + C::OFF_Q + (t + qb) * C::Q_BYTES + c * C::CHUNK_BYTES, &map_q,
                                    qf, c * 64, row0 + t * 128, bh, pol_q);
                ++q_iter;
                for (int j = 0; j < n && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        if (!mbar_wait(bar_kve(slot), phase ^ 1, ctl, kSiteKvEmpty)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar_kvf(slot), C::KV_BYTES);
                        const uint32_t dst = s_base + C::OFF_KV + slot * C::KV_BYTES;
                        for (int c = 0; c < C::KCH; ++c)
                            tma_load_3d(dst + c * C::CHUNK_BYTES, kv == 0 ? &map_k : &map_v,
                                        bar_kvf(slot), c * 64, (jlo + j) * 128, bh, pol_kv);
                        issued |= 1u << slot;
                        issued_par = (issued_par & ~(1u << slot)) | (phase << slot);
                        if (++slot == C::NSLOT) {
                            slot = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            if (*abort_flag) {  // let every load in flight land before the CTA exits
                if (SPLIT) {
                    const uint32_t f0 = (q_iter + 1) >> 1, f1 = q_iter >> 1;  // fills of buffers 0 and 1
                    if (f0 > 0) mbar_drain(BAR_QF, (f0 - 1) & 1, ctl, kSiteTeardown);
                    if (f1 > 0) mbar_drain(BAR_QF1, (f1 - 1) & 1, ctl, kSiteTeardown);
                } else if (q_iter > 0) {
                    mbar_drain(BAR_QF, (q_iter - 1) & 1, ctl, kSiteTeardown);
                }
                for (int s = 0; s < C::NSLOT; ++s)
                    if (issued & (1u << s))
                        mbar_drain(bar_kvf(s), (issued_par >> s) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        pdl_wait();  // (only its error reports touch global memory)
        if (lane == 0 && !*abort_flag) {
            int slot = 0;
            uint32_t phase = 0, q_iter = 0, p_iter = 0;
            const uint32_t sQ0 = s_base + C::OFF_Q, sQ1 = sQ0 + C::Q_BYTES;
            // one descriptor per operand per product; k-steps add constant offsets
            auto issue_s = [&](uint32_t d_col, uint32_t sQ, uint32_t sK) {
                const uint64_t a0 = sdesc_sw128(sQ, 16, 1024), b0 = sdesc_sw128(sK, 16, 1024);
                mma_ss_first(tmem + d_col, a0, b0, C::IDESC_S);
#pragma unroll
                for (int k = 1; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::CHUNK_BYTES + (k & 3) * 32;
                    mma_ss_acc(tmem + d_col, sdesc_add(a0, off), sdesc_add(b0, off), C::IDESC_S);
                }
            };
            auto issue_o = [&](uint32_t d_col, uint32_t p_col, uint32_t sV, bool acc) {
                const uint64_t b0 = sdesc_sw128(sV, C::CHUNK_BYTES, 1024);
                mma_ts(tmem + d_col, tmem + p_col, b0, C::IDESC_O, acc ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < C::BN / 16; ++k)
                    mma_ts_acc(tmem + d_col, tmem + p_col + k * 8, sdesc_add(b0, k * 2048), C::IDESC_O);
            };
            auto next = [&]() {
                if (++slot == C::NSLOT) {
                    slot = 0;
                    phase ^= 1;
                }
            };
            bool ok = true;
            uint32_t fill = 0, pit0 = 0, pit1 = 0;  // split-KV: ring fills consumed, P handoffs per warpgroup
            ItemSeq seq;
            int w_next = next_work(seq);
            SeqLen sl_next = fwd_seqlen<VL>(p, w_next);
            for (int w = w_next; w < p.num_work && ok; w = w_next) {
                w_next = next_work(seq);
                const SeqLen sl = sl_next;  // loaded one tile ahead
                sl_next = fwd_seqlen<VL>(p, w_next);
                int bh, row0;
                fwd_decode(p, w, bh, row0);
                const int n = max(0, fwd_num_kv(p, row0, sl.nq, sl.nk) - fwd_kv_first<WIN>(p, row0, sl.nq, sl.nk));
                if (n == 0) continue;
                const int qb = SPLIT ? (int)(q_iter & 1) : 0;
                const uint32_t qn = SPLIT ? (q_iter >> 1) : q_iter;
                if (!mbar_wait(qb ? BAR_QF1 : BAR_QF, qn & 1, ctl, kSiteQFull)) break;
                ++q_iter;
                if constexpr (SPLIT) {
                    // Ring fill f holds K_{f/2} (f even) or V_{f/2} (f odd) of this tile; block j goes
                    // to warpgroup j & 1, so K_{j+2} is taken before V_{j+1} (at most 3 fills ahead
                    // of the oldest one not yet released, below NSLOT).
                    const uint32_t F = fill;
                    auto fslot = [&](uint32_t f) { return (int)(f % C::NSLOT); };
                    auto fwait = [&](uint32_t f) {
                        return mbar_wait(bar_kvf(fslot(f)), (f / C::NSLOT) & 1, ctl, kSiteKvFull);
                    };
                    auto faddr = [&](uint32_t f) { return s_base + C::OFF_KV + fslot(f) * C::KV_BYTES; };
                    const uint32_t sQ = qb ? sQ1 : sQ0;
                    for (int t = 0; t < 2 && t < n; ++t) {
                        const uint32_t f = F + 2 * t;
                        if (!fwait(f)) { ok = false; break; }
                        tc_fence_after();
                        issue_s(t ? C::COL_S1 : C::COL_S0, sQ, faddr(f));
                        mma_commit(BAR_S + 8 * t);
                        mma_commit(bar_kve(fslot(f)));
                    }
                    for (int j = 0; j < n && ok; ++j) {
                        const int t = j & 1;
                        uint32_t& pit = t ? pit1 : pit0;
                        if (!mbar_wait(BAR_P + 8 * t, pit & 1, ctl, kSitePFull)) { ok = false; break; }
                        ++pit;
                        const uint32_t fv = F + 2 * j + 1;
                        if (!fwait(fv)) { ok = false; break; }
                        tc_fence_after();
                        issue_o(t ? C::COL_O1 : C::COL_O0, t ? C::COL_S1 : C::COL_S0, faddr(fv), j >= 2);
                        mma_commit(bar_kve(fslot(fv)));
                        if (j + 2 < n) {
                            const uint32_t fk = F + 2 * j + 4;
                            if (!fwait(fk)) { ok = false; break; }
                            tc_fence_after();
                            issue_s(t ? C::COL_S1 : C::COL_S0, sQ, faddr(fk));
                            mma_commit(BAR_S + 8 * t);
                            mma_commit(bar_kve(fslot(fk)));
                        } else {
                            mma_commit(BAR_O + 8 * t);
                        }
                    }
                    if (!ok) break;
                    mma_commit(qb ? BAR_QE1 : BAR_QE);
                    fill = F + 2 * n;
                    continue;
                }
                int kslot = slot;
                if (!mbar_wait(bar_kvf(kslot), phase, ctl, kSiteKvFull)) break;
                tc_fence_after();
                next();
                uint32_t sK = s_base + C::OFF_KV + kslot * C::KV_BYTES;
                issue_s(C::COL_S0, sQ0, sK);
                mma_commit(BAR_S);
                issue_s(C::COL_S1, sQ1, sK);
                mma_commit(BAR_S + 8);
                mma_commit(bar_kve(kslot));
                for (int j = 0; j < n; ++j) {
                    const int vslot = slot;
                    if (!mbar_wait(bar_kvf(vslot), phase, ctl, kSiteKvFull)) { ok = false; break; }
                    next();
                    const uint32_t sV = s_base + C::OFF_KV + vslot * C::KV_BYTES;
                    const bool more = j + 1 < n;
                    if constexpr (P_OWN) {
                        // P_t has its own columns: S_t of the next block first, then P_t V_j; the
                        // softmax learns from pv_done[t] when P_t and O_t may be written again
                        if (!mbar_wait(BAR_P, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                        tc_fence_after();
                        if (more) {
                            kslot = slot;
                            if (!mbar_wait(bar_kvf(kslot), phase, ctl, kSiteKvFull)) { ok = false; break; }
                            tc_fence_after();
                            next();
                            sK = s_base + C::OFF_KV + kslot * C::KV_BYTES;
                            issue_s(C::COL_S0, sQ0, sK);
                            mma_commit(BAR_S);
                        }
                        issue_o(C::COL_O0, C::COL_P0, sV, j > 0);
                        mma_commit(more ? BAR_PV : BAR_O);
                        if (!mbar_wait(BAR_P + 8, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                        tc_fence_after();
                        ++p_iter;
                        if (more) {
                            issue_s(C::COL_S1, sQ1, sK);
                            mma_commit(BAR_S + 8);
                            mma_commit(bar_kve(kslot));
                        }
                        issue_o(C::COL_O1, C::COL_P1, sV, j > 0);
                        mma_commit(bar_kve(vslot));
                        if (more) {
                            mma_commit(BAR_PV + 8);
                        } else {
                            mma_commit(BAR_O + 8);
                            mma_commit(BAR_QE);
                        }
                        continue;
                    }
                    if (!mbar_wait(BAR_P, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    tc_fence_after();
                    issue_o(C::COL_O0, C::COL_S0, sV, j > 0);
                    if (more) {
                        kslot = slot;
                        if (!mbar_wait(bar_kvf(kslot), phase, ctl, kSiteKvFull)) { ok = false; break; }
                        tc_fence_after();
                        next();
                        sK = s_base + C::OFF_KV + kslot * C::KV_BYTES;
                        issue_s(C::COL_S0, sQ0, sK);
                        mma_commit(BAR_S);
                    } else {
                        mma_commit(BAR_O);
                    }
                    if (!mbar_wait(BAR_P + 8, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    tc_fence_after();
                    ++p_iter;
                    issue_o(C::COL_O1, C::COL_S1, sV, j > 0);
                    mma_commit(bar_kve(vslot));
                    if (more) {
                        issue_s(C::COL_S1, sQ1, sK);
                        mma_commit(BAR_S + 8);
                        mma_commit(bar_kve(kslot));
                    } else {
                        mma_commit(BAR_O + 8);
                        mma_commit(BAR_QE);
                    }
                }
            }
            if (*abort_flag) {  // every MMA issued so far must finish before TMEM is freed
                mma_commit(BAR_TD);
                mbar_drain(BAR_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        pdl_wait();
        const int t = warp >> 2;                   // query tile of this warpgroup
        const int r = ((warp & 3) << 5) + lane;    // row within the tile = TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = t ? C::COL_S1 : C::COL_S0;
        const uint32_t col_o = t ? C::COL_O1 : C::COL_O0;
        const uint32_t bar_s = BAR_S + 8 * t, bar_p = BAR_P + 8 * t, bar_o = BAR_O + 8 * t;
        const uint32_t col_p = P_OWN ? (t ? C::COL_P1 : C::COL_P0) : col_s;
        const float c = p.scale_log2;
        uint32_t s_iter = 0, o_iter = 0, pv_iter = 0;
        uint32_t o1_iter = 0, merge_iter = 0;  // split-KV: warpgroup 1's O handoffs, merges
        bool md_pending = false;               // split-KV (warpgroup 1): merge of the last tile not yet confirmed
        float2* stage = (float2*)(smem + C::OFF_STAGE);  // split-KV: warpgroup 1's (m, l) per row
        ItemSeq seq;
        int w_next = next_work(seq);
        SeqLen sl_next = fwd_seqlen<VL>(p, w_next);
        for (int w = w_next; w < p.num_work; w = w_next) {
            w_next = next_work(seq);
            const SeqLen sl = sl_next;
            sl_next = fwd_seqlen<VL>(p, w_next);
            if (VL && sl.bad && tid == 0 && atomicCAS(&p.err->code, 0, kErrInvalid) == 0) {
                p.err->site = kSiteSeqLen;
                p.err->block = blockIdx.x;
                p.err->aux = w;
            }
            const int off = sl.nk - sl.nq;
            int bh, row0;
            fwd_decode(p, w, bh, row0);
            const int jlo = fwd_kv_first<WIN>(p, row0, sl.nq, sl.nk);
            const int n = max(0, fwd_num_kv(p, row0, sl.nq, sl.nk) - jlo);
            const int tile_row0 = row0 + (SPLIT ? 0 : t * 128);
            const int row = tile_row0 + r;
            const int j0 = SPLIT ? t : 0, jstep = SPLIT ? 2 : 1;
            float m_use = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = j0; j < n; j += jstep) {
                if (!mbar_wait(bar_s, s_iter & 1, ctl, kSiteSFull)) { ok = false; break; }
                ++s_iter;
                tc_fence_after();
                // pass 1: row maximum of the raw scores (scale > 0 commutes with max)
                const int kbase = (jlo + j) * 128;
                const bool masked = kbase + 128 > sl.nk || (p.causal && kbase + 127 > tile_row0 + off) ||
                                    (WIN && kbase < tile_row0 + 127 + off - p.window + 1) ||
                                    (VL && tile_row0 + 127 >= sl.nq);
                // last visible key of this row; none for a row past its sequence
                const int lim = (VL && row >= sl.nq) ? -1 : (p.causal ? min(row + off, sl.nk - 1) : sl.nk - 1);
                const int lim2 = lim - kbase;  // last visible column of this block
                // first visible column (sliding window), far below 0 without one
                const int lo2 = WIN ? row + off - p.window + 1 - kbase : -(1 << 30);
                // uniform over the warpgroup: masked blocks take the instantiation with the mask
                const float mraw = masked ? row_max_pass<true>(lane_addr + col_s, lim2, lo2)
                                          : row_max_pass<false>(lane_addr + col_s, lim2, lo2);
                const float m_new = fmaxf(m_use, mraw * c);
                if (P_OWN && j > j0) {  // P_t V_{j-1} must be done before O_t is rescaled or P_t rewritten
                    if (!mbar_wait(BAR_PV + 8 * t, pv_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    ++pv_iter;
                    tc_fence_after();
                }
                if (j == j0) {
                    m_use = m_new;
                } else if (__any_sync(0xffffffffu, m_new > m_use + 8.f)) {
                    // rescale the accumulator so that O and l keep a common reference max
                    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_use - m_new);
#pragma unroll 1
                    for (int q4 = 0; q4 < D / 32; ++q4) {
                        uint32_t v[32];
                        tmem_ld32(lane_addr + col_o + q4 * 32, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st32(lane_addr + col_o + q4 * 32, v);
                    }
                    l *= alpha;
                    m_use = m_new;
                }
                const float msub = (m_use == -INFINITY) ? 0.f : m_use;
                // pass 2: p = 2^(s*c - m), row sum, bf16 P over the S columns already read
                const float rsum = masked ? exp_pass<true>(lane_addr + col_s, lane_addr + col_p, lim2, lo2, c, msub)
                                          : exp_pass<false>(lane_addr + col_s, lane_addr + col_p, lim2, lo2, c, msub);
                l += rsum;
                tc_fence_before();
                if (SPLIT && md_pending) {  // O_1 is free only once the last tile's merge has read it
                    if (!mbar_wait(BAR_MD, (merge_iter - 1) & 1, ctl, kSiteOFinal)) { ok = false; break; }
                    md_pending = false;
                }
                mbar_arrive(bar_p);
            }
            if (!ok) break;
            // ---------------- epilogue: O / l -> bf16, LSE
            const int n_t = SPLIT ? (n - t + 1) / 2 : n;  // key blocks this warpgroup took
            if (n_t > 0) {
                if (!mbar_wait(bar_o, o_iter & 1, ctl, kSiteOFinal)) break;
                ++o_iter;
                tc_fence_after();
            }
            // split-KV: the other warpgroup's (m, l), and the weights of both halves
            float a0 = 1.f, a1 = 0.f;
            if constexpr (SPLIT) {
                if (t == 1) {  // hand (m, l) to warpgroup 0, which merges and stores
                    if (md_pending && !mbar_wait(BAR_MD, (merge_iter - 1) & 1, ctl, kSiteOFinal)) break;
                    stage[r] = make_float2(m_use, l);
                    tc_fence_before();
                    mbar_arrive(BAR_MR);
                    ++merge_iter;
                    md_pending = true;
                    continue;
                }
                if (!mbar_wait(BAR_MR, merge_iter & 1, ctl, kSiteOFinal)) break;
                ++merge_iter;
                const float2 ml1 = stage[r];
                if (n > 1) {  // warpgroup 1 took at least one block
                    if (!mbar_wait(BAR_O + 8, o1_iter & 1, ctl, kSiteOFinal)) break;
                    ++o1_iter;
                }
                tc_fence_after();
                if (ml1.y > 0.f) {
                    const float m = fmaxf(m_use, ml1.x);
                    a0 = (l > 0.f) ? ex2(m_use - m) : 0.f;
                    a1 = ex2(ml1.x - m);
                    l = a0 * l + a1 * ml1.y;
                    m_use = m;
                }
            }
            const bool valid = row < p.Nq;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            const float w0 = a0 * inv, w1 = a1 * inv;
            __nv_bfloat16* orow = p.o + ((size_t)bh * p.Nq + (valid ? row : 0)) * D;
            const bool o_wide = ((uintptr_t)p.o & 31) == 0;  // rows are 32-byte multiples
#pragma unroll 1
            for (int q4 = 0; q4 < D / 32; ++q4) {
                uint32_t v[32];
                if (n > 0) {
                    tmem_ld32(lane_addr + col_o + q4 * 32, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
                uint32_t pk[16];
                // tcgen05.ld is warp-collective: the O_1 read depends on the tile (n), never on the
                // row; rows whose half 1 saw no key have a1 = 0 and O_1 = 0 there.
                if (SPLIT && n > 1) {
                    uint32_t u[32];
                    tmem_ld32(lane_addr + C::COL_O1 + q4 * 32, u);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * w0 + __uint_as_float(u[2 * i]) * w1,
                                          __uint_as_float(v[2 * i + 1]) * w0 + __uint_as_float(u[2 * i + 1]) * w1);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * w0, __uint_as_float(v[2 * i + 1]) * w0);
                }
                if (valid) store_row64(orow + q4 * 32, pk, o_wide);
            }
            if (valid)
                p.lse[(size_t)bh * p.Nq + row] =
                    (l > 0.f) ? (m_use + lg2(l)) * 0.69314718055994531f : -INFINITY;
            tc_fence_before();
            if (SPLIT) mbar_arrive(BAR_MD);  // O_1 and the staged (m, l) may be overwritten
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) {
        __syncwarp();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Heads per scheduling chunk: their K and V fit in 64 MiB of L2 together.
// Causal and non-causal alike: causal grids take the chunks in per-chunk
// rounds (next_chunked_item), so their tiles' weights still even out per CTA.
int fwd_head_chunk(int BH, int Nk, int d) {
    const long long per_head = 4ll * Nk * d;
    return (int)std::max(1ll, std::min((long long)BH, (64ll << 20) / per_head));
}

template <int D, bool WIN, bool VL, bool SPLIT>
cudaError_t launch_fwd_dw(const FwdLaunch& a, cudaStream_t s) {
    using C = Fwd<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    static_assert(!SPLIT || !VL, "split-KV tiles are built for the plain and the window forward only");
    cudaError_t e = set_smem_limit_once<fwd_kernel<D, WIN, VL, SPLIT>>(C::SMEM);
    if (e != cudaSuccess) return e;
    FwdParams p;
    p.o = (__nv_bfloat16*)a.o;
    p.lse = a.lse;
    p.BH = a.B * a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.causal = a.causal;
    p.window = a.window;
    p.lens_q = a.lens_q;
    p.lens_k = a.lens_k;
    p.H = a.H;
    p.rows = SPLIT ? 128 : kFwdRowsPerCta;
    p.n_mtiles = (a.Nq + p.rows - 1) / p.rows;
    // chunks of heads whose K and V fit in 64 MiB of L2 together (split-KV grids are small: one chunk)
    if (SPLIT) {
        p.hc = p.BH;
        p.per_chunk = 0;
    } else {
        fwd_work_order(p.BH, a.Nq, a.Nk, a.causal, fwd_head_chunk(p.BH, a.Nk, a.d), a.num_sms, &p.hc, &p.per_chunk);
    }
    p.num_work = p.n_mtiles * p.BH;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    p.timeout_ns = a.timeout_ns;
    const int grid = p.num_work < a.num_sms ? p.num_work : a.num_sms;
    return launch_dependent(fwd_kernel<D, WIN, VL, SPLIT>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, s, a.map_q,
                            a.map_k, a.map_v, p);
}

// Tile mode for the plain forward.  The grid is persistent with a static
// schedule (next_chunked_item), so the host can add up every CTA's share for
// both tile sizes and take the one whose busiest CTA finishes first.  Costs, in units of one 128-key block of
// a 256-row tile, fitted to GB300 timings: a key block of a split-KV tile
// costs 0.55 (half the rows, but the two softmax warpgroups alternate on one
// tile's blocks, at ~85% of the two-tile rate), and a tile costs 1.5 (256
// rows) or 2 (split-KV: the merge) for its prologue and epilogue.  Only small
// grids are evaluated; past four tiles per SM the 256-row tiles always win.
int fwd_makespan(int BH, int Nq, int Nk, int causal, int rows, int hc, bool per_chunk, int block_cost, int tile_cost,
                 int num_sms) {
    const int n_m = (Nq + rows - 1) / rows;
    const int work = n_m * BH, G = work < num_sms ? work : num_sms;
    const int kv_total = (Nk + 127) / 128;
    long long mx = 0;
    for (int c = 0; c < G; ++c) {
        long long tot = 0;
        ItemSeq q;
        for (int w = next_chunked_item(q, work, hc * n_m, G, c, per_chunk); w < work;
             w = next_chunked_item(q, work, hc * n_m, G, c, per_chunk)) {
            const int chunk = w / (hc * n_m), r = w - chunk * hc * n_m;
            const int hn = hc < BH - chunk * hc ? hc : BH - chunk * hc;
            const int mr = r / hn, m = causal ? n_m - 1 - mr : mr;
            int n = kv_total;
            if (causal) {
                const long long lim = (long long)(m * rows + rows - 1 < Nq - 1 ? m * rows + rows - 1 : Nq - 1) + Nk - Nq;
                n = lim < 0 ? 0 : (int)(lim / 128 + 1 < kv_total ? lim / 128 + 1 : kv_total);
            }
            tot += (long long)n * block_cost + tile_cost;
        }
        mx = tot > mx ? tot : mx;
    }
    return (int)(mx < (1LL << 30) ? mx : (1LL << 30));
}

template <int D>
cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t s) {
    if (a.lens_q || a.lens_k) return launch_fwd_dw<D, false, true, false>(a, s);
    // a window of at most 129 keys (a 128-row tile then sees at most two key blocks when Nk - Nq is a
    // multiple of 128): split-KV tiles (each warpgroup takes every other block of a 128-row tile) halve
    // the chain per tile, whose fixed costs dominate at so few blocks per tile
    if (a.window > 0)
        return a.window <= 129 ? launch_fwd_dw<D, true, false, true>(a, s) : launch_fwd_dw<D, true, false, false>(a, s);
    return fwd_use_split(a) ? launch_fwd_dw<D, false, false, true>(a, s) : launch_fwd_dw<D, false, false, false>(a, s);
}

}  // namespace

bool fwd_use_split(const FwdLaunch& a) {
    const long long work256 = (long long)((a.Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta) * a.B * a.H;
    if (work256 > 4LL * a.num_sms || a.num_sms > 1024 || a.num_sms <= 0) return false;
    const int BH = a.B * a.H;
    int hc, per_chunk;
    fwd_work_order(BH, a.Nq, a.Nk, a.causal, fwd_head_chunk(BH, a.Nk, a.d), a.num_sms, &hc, &per_chunk);
    return fwd_makespan(BH, a.Nq, a.Nk, a.causal, 128, BH, false, 55, 200, a.num_sms) <
           fwd_makespan(BH, a.Nq, a.Nk, a.causal, kFwdRowsPerCta, hc, per_chunk != 0, 100, 150, a.num_sms);
}

void fwd_work_order(int BH, int Nq, int Nk, int causal, int hc_l2, int num_sms, int* hc, int* per_chunk) {
    *hc = hc_l2;
    *per_chunk = causal ? 1 : 0;
    if (!causal || hc_l2 >= BH || num_sms <= 0) return;
    // past ~1M work tiles the replay would cost milliseconds of host time per new shape; the
    // chunks' remainders are a smaller share there, so the chunked order stays
    if ((long long)((Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta) * BH > (1ll << 20)) return;
    // The one-chunk order's rounds pair heavy and light tiles exactly; per-chunk rounds leave each
    // chunk's remainder (up to ~2% at N >= 16384) and are kept when within 0.5% of it.  The replay
    // walks every tile once per schedule, so the last shape's answer is kept.
    static std::mutex mu;
    static long long last_key[6] = {-1, -1, -1, -1, -1, -1};
    static int last_hc = 0;
    const long long key[6] = {BH, Nq, Nk, hc_l2, num_sms, 1};
    std::lock_guard<std::mutex> lock(mu);
    if (std::equal(key, key + 6, last_key)) {
        *hc = last_hc;
        return;
    }
    const long long chunked = fwd_makespan(BH, Nq, Nk, 1, kFwdRowsPerCta, hc_l2, true, 100, 150, num_sms);
    const long long one = fwd_makespan(BH, Nq, Nk, 1, kFwdRowsPerCta, BH, true, 100, 150, num_sms);
    if (chunked * 1000 > one * 1005) *hc = BH;
    std::copy(key, key + 6, last_key);
    last_hc = *hc;
}

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_fwd_d<128>(a, s) : launch_fwd_d<64>(a, s);
}

}  // namespace fa
