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
    // barriers: q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], o_final[2], teardown
    static constexpr int NBAR = 2 + 2 * NSLOT + 7;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
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
    int n_mtiles, num_work;
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
    const int max_row = min(row0 + kFwdRowsPerCta - 1, nq - 1);
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

// Work tile w -> (bh, first row).  Causal: heaviest row tiles first.
__device__ __forceinline__ void fwd_decode(const FwdParams& p, int w, int& bh, int& row0) {
    const int mr = w / p.BH;
    bh = w - mr * p.BH;
    const int m = p.causal ? (p.n_mtiles - 1 - mr) : mr;
    row0 = m * kFwdRowsPerCta;
}

// Pass 1 over one 128-column S row in TMEM (thread = row): the maximum of the
// raw scores.  Chunks of 32 columns are double-buffered (the next loads while
// this one is scanned).  MASKED: columns c > lim2 or c < lo2 are excluded;
// instantiated only for the blocks that hold a masked column.
template <bool MASKED>
__device__ __forceinline__ float row_max_pass(uint32_t taddr, int lim2, int lo2) {
    float mraw = -INFINITY;
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
            mraw = fmax3(mraw, x0, x1);
        }
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    return mraw;
}

// Pass 2: p = 2^(s c - m) for the 128 columns, their sum, and bf16 P written
// over the S columns already read (keys [32 q, 32 q + 32) to columns
// [16 q, 16 q + 16); the load in flight is always of columns >= 32 (q + 1)).
template <bool MASKED>
__device__ __forceinline__ float exp_pass(uint32_t taddr, int lim2, int lo2, float c, float msub) {
    float2 rs = make_float2(0.f, 0.f);
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
            rs = fadd2(rs, e);
            pk[i] = pack_bf16(e.x, e.y);
        }
        tmem_st16_async(taddr + q4 * 16, pk);
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    tmem_wait_st();
    return rs.x + rs.y;
}

// WIN: the sliding-window variant; VL: per-sequence lengths (rows past a
// sequence's length give O = 0, LSE = -inf; keys past it are masked).  Each is
// a separate instantiation, so the plain path carries none of their bounds.
template <int D, bool WIN, bool VL>
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
    uint32_t* tmem_slot = (uint32_t*)(smem + C::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int slot = 0;
            uint32_t phase = 0, q_iter = 0;
            uint32_t issued = 0, issued_par = 0;  // per slot: filled at least once / its last parity
            bool ok = true;
            SeqLen sl_next = fwd_seqlen<VL>(p, persistent_work(0, blockIdx.x, gridDim.x));
            for (int rd = 0; rd * (int)gridDim.x < p.num_work && ok; ++rd) {
                const int w = persistent_work(rd, blockIdx.x, gridDim.x);
                const SeqLen sl = sl_next;  // loaded one tile ahead
                sl_next = fwd_seqlen<VL>(p, persistent_work(rd + 1, blockIdx.x, gridDim.x));
                if (w >= p.num_work) continue;
                int bh, row0;
                fwd_decode(p, w, bh, row0);
                const int jlo = fwd_kv_first<WIN>(p, row0, sl.nq, sl.nk);
                const int n = max(0, fwd_num_kv(p, row0, sl.nq, sl.nk) - jlo);
                if (n == 0) continue;
                if (q_iter > 0 && !mbar_wait(BAR_QE, (q_iter - 1) & 1, ctl, kSiteQEmpty)) break;
                mbar_arrive_expect_tx(BAR_QF, 2 * C::Q_BYTES);
                for (int t = 0; t < 2; ++t)
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_3d(s_base + C::OFF_Q + t * C::Q_BYTES + c * C::CHUNK_BYTES, &map_q,
                                    BAR_QF, c * 64, row0 + t * 128, bh, pol_q);
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
                if (q_iter > 0) mbar_drain(BAR_QF, (q_iter - 1) & 1, ctl, kSiteTeardown);
                for (int s = 0; s < C::NSLOT; ++s)
                    if (issued & (1u << s))
                        mbar_drain(bar_kvf(s), (issued_par >> s) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag) {
            int slot = 0;
            uint32_t phase = 0, q_iter = 0, p_iter = 0;
            const uint32_t sQ0 = s_base + C::OFF_Q, sQ1 = sQ0 + C::Q_BYTES;
            auto issue_s = [&](uint32_t d_col, uint32_t sQ, uint32_t sK) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::CHUNK_BYTES + (k & 3) * 32;
                    mma_ss(tmem + d_col, sdesc_sw128(sQ + off, 16, 1024),
                           sdesc_sw128(sK + off, 16, 1024), C::IDESC_S, k > 0);
                }
            };
            auto issue_o = [&](uint32_t d_col, uint32_t p_col, uint32_t sV, bool acc) {
#pragma unroll
                for (int k = 0; k < C::BN / 16; ++k)
                    mma_ts(tmem + d_col, tmem + p_col + k * 8,
                           sdesc_sw128(sV + k * 2048, C::CHUNK_BYTES, 1024), C::IDESC_O,
                           (acc || k > 0) ? 1u : 0u);
            };
            auto next = [&]() {
                if (++slot == C::NSLOT) {
                    slot = 0;
                    phase ^= 1;
                }
            };
            bool ok = true;
            SeqLen sl_next = fwd_seqlen<VL>(p, persistent_work(0, blockIdx.x, gridDim.x));
            for (int rd = 0; rd * (int)gridDim.x < p.num_work && ok; ++rd) {
                const int w = persistent_work(rd, blockIdx.x, gridDim.x);
                const SeqLen sl = sl_next;  // loaded one tile ahead
                sl_next = fwd_seqlen<VL>(p, persistent_work(rd + 1, blockIdx.x, gridDim.x));
                if (w >= p.num_work) continue;
                int bh, row0;
                fwd_decode(p, w, bh, row0);
                const int n = max(0, fwd_num_kv(p, row0, sl.nq, sl.nk) - fwd_kv_first<WIN>(p, row0, sl.nq, sl.nk));
                if (n == 0) continue;
                if (!mbar_wait(BAR_QF, q_iter & 1, ctl, kSiteQFull)) break;
                ++q_iter;
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
        const int t = warp >> 2;                   // query tile of this warpgroup
        const int r = ((warp & 3) << 5) + lane;    // row within the tile = TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = t ? C::COL_S1 : C::COL_S0;
        const uint32_t col_o = t ? C::COL_O1 : C::COL_O0;
        const uint32_t bar_s = BAR_S + 8 * t, bar_p = BAR_P + 8 * t, bar_o = BAR_O + 8 * t;
        const float c = p.scale_log2;
        uint32_t s_iter = 0, o_iter = 0;
        SeqLen sl_next = fwd_seqlen<VL>(p, persistent_work(0, blockIdx.x, gridDim.x));
        for (int rd = 0; rd * (int)gridDim.x < p.num_work; ++rd) {
            const int w = persistent_work(rd, blockIdx.x, gridDim.x);
            const SeqLen sl = sl_next;
            sl_next = fwd_seqlen<VL>(p, persistent_work(rd + 1, blockIdx.x, gridDim.x));
            if (w >= p.num_work) continue;
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
            const int tile_row0 = row0 + t * 128;
            const int row = tile_row0 + r;
            float m_use = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < n; ++j) {
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
                if (j == 0) {
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
                const float rsum = masked ? exp_pass<true>(lane_addr + col_s, lim2, lo2, c, msub)
                                          : exp_pass<false>(lane_addr + col_s, lim2, lo2, c, msub);
                l += rsum;
                tc_fence_before();
                mbar_arrive(bar_p);
            }
            if (!ok) break;
            // ---------------- epilogue: O / l -> bf16, LSE
            if (n > 0) {
                if (!mbar_wait(bar_o, o_iter & 1, ctl, kSiteOFinal)) break;
                ++o_iter;
                tc_fence_after();
            }
            const bool valid = row < p.Nq;
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            __nv_bfloat16* orow = p.o + ((size_t)bh * p.Nq + (valid ? row : 0)) * D;
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
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
            if (valid)
                p.lse[(size_t)bh * p.Nq + row] =
                    (l > 0.f) ? (m_use + lg2(l)) * 0.69314718055994531f : -INFINITY;
            tc_fence_before();
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

template <int D, bool WIN, bool VL>
cudaError_t launch_fwd_dw(const FwdLaunch& a, cudaStream_t s) {
    using C = Fwd<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, WIN, VL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
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
    p.n_mtiles = (a.Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta;
    p.num_work = p.n_mtiles * p.BH;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    p.timeout_ns = a.timeout_ns;
    const int grid = p.num_work < a.num_sms ? p.num_work : a.num_sms;
    fwd_kernel<D, WIN, VL><<<grid, C::THREADS, C::SMEM, s>>>(a.map_q, a.map_k, a.map_v, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t s) {
    if (a.lens_q || a.lens_k) return launch_fwd_dw<D, false, true>(a, s);
    return a.window > 0 ? launch_fwd_dw<D, true, false>(a, s) : launch_fwd_dw<D, false, false>(a, s);
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_fwd_d<128>(a, s) : launch_fwd_d<64>(a, s);
}

}  // namespace fa
