// FP8 (e4m3) forward with block scales (d = 128).
//
// The method is the forward of fa_fwd.cu (wiki.ai-engineering.at "Flash
// Attention", "Tiling Algorithm" and "Lösung: Online Softmax"), with the
// operands in 8-bit floating point, the block-scaled attention that
// johe.ru "Flash Attention: ...", section "Flash Attention 3", lists among
// its optimisations, and the FP8 support of its "Flash Attention 4" section.
// Inputs: Q and K in e4m3 with one fp32 scale per 128-row block (the value of
// an element is its e4m3 value times its block's scale), V in e4m3 with one
// fp32 scale per head.  Per tile pair the score scale is scale * sq_i * sk_j,
// folded into the softmax constant; P is rounded to e4m3 for the value
// product, whose result is multiplied by the head's V scale in the epilogue.
//
// GB300 mapping: the fa_fwd.cu structure (persistent CTA, 320 threads, two
// 128-row query tiles per work tile, MMA warp 9, TMA producer warp 8, one
// softmax warpgroup per query tile) with kind::f8f6f4 products:
//   S_t = Q_t K_j^T    M = 128, N = 128, K = 128 (4 steps of 32 bytes)
//   O_t += P_t V_j     P_t from shared memory (the softmax threads write their
//                      row as e4m3, 128-byte swizzle), V_j^T from a transposed
//                      copy of V (both operands K-major).
// Since P_t does not alias S_t, S_t(j+1) is issued ahead of P_t V_j; a
// pv_done[t] barrier tells the softmax when P_t and O_t may be written again.
// The transposed copy [B*H, 128, Nk rounded up to 16] is made by vt_kernel into
// the caller's workspace before the forward runs.
#include <algorithm>

#include "fa_internal.h"

namespace fa {
namespace {

struct F8 {
    static constexpr int D = 128;
    static constexpr int TILE = 128 * 128;      // 128 rows x 128 bytes: one swizzle atom wide
    static constexpr int NSLOT = 8;             // K and V^T tiles in flight
    static constexpr int OFF_Q = 0;             // query tiles t = 0, 1
    static constexpr int OFF_P = 2 * TILE;      // P tiles t = 0, 1
    static constexpr int OFF_KV = 4 * TILE;
    static constexpr int OFF_BAR = OFF_KV + NSLOT * TILE;
    // q_full, q_empty, kv_full[NSLOT], kv_empty[NSLOT], s_full[2], p_full[2], o_final[2], teardown,
    // pv_done[2]
    static constexpr int NBAR = 2 + 2 * NSLOT + 9;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
};
static_assert(F8::SMEM <= 232448, "shared memory budget");

// Instruction descriptor of kind::f8f6f4: D fp32, A and B e4m3 (format 0), both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescF8 = idesc_e4m3(128, 128);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdescF8), "r"(accumulate)
        : "memory");
}
// The same with the accumulate flag fixed on (every k-step after the first).
__device__ __forceinline__ void mma_f8_acc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc) {
    asm volatile("tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, 1;" ::"r"(d_tmem), "l"(adesc),
                 "l"(bdesc), "r"(kIdescF8)
                 : "memory");
}

// Four fp32 values -> four e4m3 bytes (x0 in the lowest byte), round to nearest
// even, saturating at the largest finite value.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

struct F8Params {
    __nv_bfloat16* o;
    float* lse;
    const float* q_scale;  // [B*H, ceil(Nq/128)]
    const float* k_scale;  // [B*H, ceil(Nk/128)]
    const float* v_scale;  // [B*H]
    int hc;  // heads per scheduling chunk
    int per_chunk;  // the CTAs take the chunks in per-chunk rounds (next_chunked_item)
    int BH, Nq, Nk, causal, n_qb, n_kb;
    int n_mtiles, num_work;
    float scale_log2;
    DevError* err;
    uint64_t timeout_ns;
};

__device__ __forceinline__ int f8_num_kv(const F8Params& p, int row0) {
    const int kv_total = (p.Nk + 127) / 128;
    if (!p.causal) return kv_total;
    const int max_row = min(row0 + kFwdRowsPerCta - 1, p.Nq - 1);
    const long long lim = (long long)max_row + p.Nk - p.Nq;
    if (lim < 0) return 0;
    return min(kv_total, (int)(lim / 128) + 1);
}

// Work tile w -> (bh, first row), as the bf16 forward's: heads in chunks of hc
// whose K and V fit in L2 together, every head's row tile of one level before
// the next level within a chunk (causal: heaviest first).
__device__ __forceinline__ void f8_decode(const F8Params& p, int w, int& bh, int& row0) {
    const int chunk = p.hc * p.n_mtiles;
    const int c = w / chunk;
    const int r = w - c * chunk;
    const int h0 = c * p.hc;
    const int hn = min(p.hc, p.BH - h0);
    const int mr = r / hn;
    bh = h0 + (r - mr * hn);
    const int m = p.causal ? (p.n_mtiles - 1 - mr) : mr;
    row0 = m * kFwdRowsPerCta;
}

// Row maximum of the raw scores of one 128-column S row (thread = row).
template <bool MASKED>
__device__ __forceinline__ float f8_row_max(uint32_t taddr, int lim2) {
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
                if (q4 * 32 + i > lim2) x0 = -INFINITY;
                if (q4 * 32 + i + 1 > lim2) x1 = -INFINITY;
            }
            mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x0, x1);
        }
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
}

// p = 2^(s c - m) for the 128 columns, their sum, and P as e4m3 into the
// thread's row of the P tile (16-byte granule g at g ^ (r & 7)).
template <bool MASKED>
__device__ __forceinline__ float f8_exp_row(uint32_t taddr, int lim2, float c, float msub, uint8_t* prow, int r) {
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
        uint32_t pk[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            float e[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                const int col = q4 * 32 + 4 * w + u;
                float s0 = __uint_as_float(v[4 * w + u]), s1 = __uint_as_float(v[4 * w + u + 1]);
                if constexpr (MASKED) {
                    if (col > lim2) s0 = -INFINITY;
                    if (col + 1 > lim2) s1 = -INFINITY;
                }
                const float2 x = ffma2(make_float2(s0, s1), c2, nm2);
                e[u] = ex2(x.x);
                e[u + 1] = ex2(x.y);
                rs[(2 * w + u / 2) & 3] = fadd2(rs[(2 * w + u / 2) & 3], make_float2(e[u], e[u + 1]));
            }
            pk[w] = pack_e4m3x4(e[0], e[1], e[2], e[3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int g = q4 * 2 + h;
            *reinterpret_cast<uint4*>(prow + ((g ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
        }
        if (q4 + 1 < 4) tmem_wait_ld(nx);
    }
    const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
    return (r01.x + r23.x) + (r01.y + r23.y);
}

__global__ void __launch_bounds__(F8::THREADS, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_vt, const F8Params p) {
    using C = F8;
    constexpr int D = C::D;
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
    const uint32_t BAR_PV = BAR_TD + 8;               // pv_done[t]: P_t V_j done (P_t and O_t free again)
    uint32_t* tmem_slot = (uint32_t*)(smem + C::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's work tiles (every role walks the same sequence; next_chunked_item)
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
        mbar_init(BAR_PV, 1);
        mbar_init(BAR_PV + 8, 1);
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
    pdl_launch_dependents();
    pdl_wait();  // the setup above overlaps the V transpose; its V^T is visible from here

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            tma_prefetch_desc(&map_q);
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_vt);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int slot = 0;
            uint32_t phase = 0, q_iter = 0, issued = 0, issued_par = 0;
            bool ok = true;
            ItemSeq seq;
            for (int w = next_work(seq); w < p.num_work && ok; w = next_work(seq)) {
                int bh, row0;
                f8_decode(p, w, bh, row0);
                const int n = f8_num_kv(p, row0);
                if (n == 0) continue;
                if (q_iter > 0 && !mbar_wait(BAR_QE, (q_iter - 1) & 1, ctl, kSiteQEmpty)) break;
                mbar_arrive_expect_tx(BAR_QF, 2 * C::TILE);
                for (int t = 0; t < 2; ++t)
                    tma_load_3d(s_base + C::OFF_Q + t * C::TILE, &map_q, BAR_QF, 0, row0 + t * 128, bh, pol_q);
                ++q_iter;
                for (int j = 0; j < n && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        if (!mbar_wait(bar_kve(slot), phase ^ 1, ctl, kSiteKvEmpty)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar_kvf(slot), C::TILE);
                        const uint32_t dst = s_base + C::OFF_KV + slot * C::TILE;
                        if (kv == 0)
                            tma_load_3d(dst, &map_k, bar_kvf(slot), 0, j * 128, bh, pol_kv);
                        else  // V^T tile: keys [128 j, 128 j + 128) of all 128 feature rows
                            tma_load_3d(dst, &map_vt, bar_kvf(slot), j * 128, 0, bh, pol_kv);
                        issued |= 1u << slot;
                        issued_par = (issued_par & ~(1u << slot)) | (phase << slot);
                        if (++slot == C::NSLOT) {
                            slot = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            if (*abort_flag) {
                if (q_iter > 0) mbar_drain(BAR_QF, (q_iter - 1) & 1, ctl, kSiteTeardown);
                for (int s = 0; s < C::NSLOT; ++s)
                    if (issued & (1u << s)) mbar_drain(bar_kvf(s), (issued_par >> s) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort_flag) {
            int slot = 0;
            uint32_t phase = 0, q_iter = 0, p_iter = 0;
            const uint32_t sQ0 = s_base + C::OFF_Q, sQ1 = sQ0 + C::TILE;
            const uint32_t sP0 = s_base + C::OFF_P, sP1 = sP0 + C::TILE;
            // A and B both K-major, 128-byte rows: K step k starts 32 k bytes into the rows
            // one descriptor per operand per product; k-steps add constant offsets
            auto issue_s = [&](uint32_t d_col, uint32_t sQ, uint32_t sK) {
                const uint64_t a0 = sdesc_sw128(sQ, 16, 1024), b0 = sdesc_sw128(sK, 16, 1024);
                mma_f8(tmem + d_col, a0, b0, 0u);
#pragma unroll
                for (int k = 1; k < D / 32; ++k) mma_f8_acc(tmem + d_col, sdesc_add(a0, 32 * k), sdesc_add(b0, 32 * k));
            };
            auto issue_o = [&](uint32_t d_col, uint32_t sP, uint32_t sVt, bool acc) {
                const uint64_t a0 = sdesc_sw128(sP, 16, 1024), b0 = sdesc_sw128(sVt, 16, 1024);
                mma_f8(tmem + d_col, a0, b0, acc ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < 128 / 32; ++k)
                    mma_f8_acc(tmem + d_col, sdesc_add(a0, 32 * k), sdesc_add(b0, 32 * k));
            };
            auto next = [&]() {
                if (++slot == C::NSLOT) {
                    slot = 0;
                    phase ^= 1;
                }
            };
            bool ok = true;
            ItemSeq seq;
            for (int w = next_work(seq); w < p.num_work && ok; w = next_work(seq)) {
                int bh, row0;
                f8_decode(p, w, bh, row0);
                const int n = f8_num_kv(p, row0);
                if (n == 0) continue;
                if (!mbar_wait(BAR_QF, q_iter & 1, ctl, kSiteQFull)) break;
                ++q_iter;
                int kslot = slot;
                if (!mbar_wait(bar_kvf(kslot), phase, ctl, kSiteKvFull)) break;
                tc_fence_after();
                next();
                uint32_t sK = s_base + C::OFF_KV + kslot * C::TILE;
                issue_s(C::COL_S0, sQ0, sK);
                mma_commit(BAR_S);
                issue_s(C::COL_S1, sQ1, sK);
                mma_commit(BAR_S + 8);
                mma_commit(bar_kve(kslot));
                // Per block j and tile t: S_t(j+1) first, then P_t V_j.  P_t lives in shared
                // memory, not over S_t, so the next scores need not wait for the value product;
                // the softmax learns from pv_done[t] when P_t and O_t may be written again.
                for (int j = 0; j < n; ++j) {
                    const int vslot = slot;
                    if (!mbar_wait(bar_kvf(vslot), phase, ctl, kSiteKvFull)) { ok = false; break; }
                    next();
                    const uint32_t sVt = s_base + C::OFF_KV + vslot * C::TILE;
                    const bool more = j + 1 < n;
                    if (!mbar_wait(BAR_P, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    tc_fence_after();
                    if (more) {
                        kslot = slot;
                        if (!mbar_wait(bar_kvf(kslot), phase, ctl, kSiteKvFull)) { ok = false; break; }
                        tc_fence_after();
                        next();
                        sK = s_base + C::OFF_KV + kslot * C::TILE;
                        issue_s(C::COL_S0, sQ0, sK);
                        mma_commit(BAR_S);
                    }
                    issue_o(C::COL_O0, sP0, sVt, j > 0);
                    mma_commit(more ? BAR_PV : BAR_O);
                    if (!mbar_wait(BAR_P + 8, p_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    tc_fence_after();
                    ++p_iter;
                    if (more) {
                        issue_s(C::COL_S1, sQ1, sK);
                        mma_commit(BAR_S + 8);
                        mma_commit(bar_kve(kslot));
                    }
                    issue_o(C::COL_O1, sP1, sVt, j > 0);
                    mma_commit(bar_kve(vslot));
                    if (more) {
                        mma_commit(BAR_PV + 8);
                    } else {
                        mma_commit(BAR_O + 8);
                        mma_commit(BAR_QE);
                    }
                }
            }
            if (*abort_flag) {
                mma_commit(BAR_TD);
                mbar_drain(BAR_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = t ? C::COL_S1 : C::COL_S0;
        const uint32_t col_o = t ? C::COL_O1 : C::COL_O0;
        const uint32_t bar_s = BAR_S + 8 * t, bar_p = BAR_P + 8 * t, bar_o = BAR_O + 8 * t;
        const uint32_t bar_pv = BAR_PV + 8 * t;
        uint8_t* prow = smem + C::OFF_P + t * C::TILE + r * 128;
        const int off = p.Nk - p.Nq;
        uint32_t s_iter = 0, o_iter = 0, pv_iter = 0;
        ItemSeq seq;
        for (int w = next_work(seq); w < p.num_work; w = next_work(seq)) {
            int bh, row0;
            f8_decode(p, w, bh, row0);
            const int n = f8_num_kv(p, row0);
            const int tile_row0 = row0 + t * 128;
            const int row = tile_row0 + r;
            const int qb = min(tile_row0 / 128, p.n_qb - 1);
            const float cq = p.scale_log2 * __ldg(p.q_scale + (size_t)bh * p.n_qb + qb);
            const float* ks = p.k_scale + (size_t)bh * p.n_kb;
            float sk_next = n > 0 ? __ldg(ks) : 0.f;
            float m_use = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < n; ++j) {
                const float c = cq * sk_next;  // this block's score constant
                if (j + 1 < n) sk_next = __ldg(ks + j + 1);
                if (!mbar_wait(bar_s, s_iter & 1, ctl, kSiteSFull)) { ok = false; break; }
                ++s_iter;
                tc_fence_after();
                const int kbase = j * 128;
                const bool masked = kbase + 128 > p.Nk || (p.causal && kbase + 127 > tile_row0 + off);
                const int lim = p.causal ? min(row + off, p.Nk - 1) : p.Nk - 1;
                const int lim2 = lim - kbase;
                const float mraw = masked ? f8_row_max<true>(lane_addr + col_s, lim2)
                                          : f8_row_max<false>(lane_addr + col_s, lim2);
                const float m_new = fmaxf(m_use, mraw * c);
                if (j > 0) {  // P_t V_{j-1} must be done before O_t is rescaled or P_t rewritten
                    if (!mbar_wait(bar_pv, pv_iter & 1, ctl, kSitePFull)) { ok = false; break; }
                    ++pv_iter;
                    tc_fence_after();
                }
                if (j == 0) {
                    m_use = m_new;
                } else if (__any_sync(0xffffffffu, m_new > m_use + 8.f)) {
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
                const float rsum = masked ? f8_exp_row<true>(lane_addr + col_s, lim2, c, msub, prow, r)
                                          : f8_exp_row<false>(lane_addr + col_s, lim2, c, msub, prow, r);
                l += rsum;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P tile -> tensor core
                tc_fence_before();
                mbar_arrive(bar_p);
            }
            if (!ok) break;
            if (n > 0) {
                if (!mbar_wait(bar_o, o_iter & 1, ctl, kSiteOFinal)) break;
                ++o_iter;
                tc_fence_after();
            }
            const bool valid = row < p.Nq;
            const float inv = (l > 0.f) ? __ldg(p.v_scale + bh) / l : 0.f;
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
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
                if (valid) store_row64(orow + q4 * 32, pk, o_wide);
            }
            if (valid)
                p.lse[(size_t)bh * p.Nq + row] = (l > 0.f) ? (m_use + lg2(l)) * 0.69314718055994531f : -INFINITY;
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

// V [BH, Nk, 128] e4m3 -> V^T [BH, 128, Nk_pad] (keys past Nk are zero).
// One CTA per (head, 128-key block): a 128 x 128 byte tile through shared
// memory as 32-bit words.  Each thread then transposes 4 x 4 byte blocks with
// byte permutes: 16 keys of 4 features, written as four 16-byte pieces of V^T
// rows; the 8 threads sharing a feature word cover 128 contiguous keys.
__global__ void __launch_bounds__(256) vt_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt, int Nk,
                                                 int Nk_pad) {
    // [key][feature word]: word w of key k sits in column (w + 4 (k / 16)) mod 32 of a 33-word row, which keeps
    // both the row-wise fill and the column-wise read free of bank conflicts.
    __shared__ uint32_t tw[128][33];
    const int bh = blockIdx.x, kb = blockIdx.y, tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();  // V may come from the kernel before, which may still read the workspace
    const uint8_t* src = v + (size_t)bh * Nk * 128;
    for (int i = tid; i < 128 * 8; i += 256) {  // 128 keys x 8 granules of 16 bytes
        const int key = i >> 3, g = i & 7, rot = 4 * (key >> 4);
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (kb * 128 + key < Nk) x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(kb * 128 + key) * 128) + g);
        tw[key][(4 * g + rot) & 31] = x.x;
        tw[key][(4 * g + 1 + rot) & 31] = x.y;
        tw[key][(4 * g + 2 + rot) & 31] = x.z;
        tw[key][(4 * g + 3 + rot) & 31] = x.w;
    }
    __syncthreads();
    const int kg = tid & 7, fw = tid >> 3;  // keys 16 kg .. 16 kg + 15 of the tile, features 4 fw .. 4 fw + 3
    const int key0 = kb * 128 + kg * 16, col = (fw + 4 * kg) & 31;
    if (key0 >= Nk_pad) return;
    uint32_t out[4][4];  // [feature][4 keys]
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int k = kg * 16 + 4 * q;
        const uint32_t a = tw[k][col], b = tw[k + 1][col], c = tw[k + 2][col], d = tw[k + 3][col];
        const uint32_t ab_lo = __byte_perm(a, b, 0x5140), ab_hi = __byte_perm(a, b, 0x7362);  // a0 b0 a1 b1 / a2 b2 a3 b3
        const uint32_t cd_lo = __byte_perm(c, d, 0x5140), cd_hi = __byte_perm(c, d, 0x7362);
        out[0][q] = __byte_perm(ab_lo, cd_lo, 0x5410);  // a0 b0 c0 d0
        out[1][q] = __byte_perm(ab_lo, cd_lo, 0x7632);  // a1 b1 c1 d1
        out[2][q] = __byte_perm(ab_hi, cd_hi, 0x5410);
        out[3][q] = __byte_perm(ab_hi, cd_hi, 0x7632);
    }
    uint8_t* dst = vt + (size_t)bh * 128 * Nk_pad + key0;
#pragma unroll
    for (int f = 0; f < 4; ++f)
        *reinterpret_cast<uint4*>(dst + (size_t)(4 * fw + f) * Nk_pad) = make_uint4(out[f][0], out[f][1], out[f][2], out[f][3]);
}

}  // namespace

cudaError_t launch_fwd_fp8(const Fp8FwdLaunch& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    if ((a.Nk_pad + 127) / 128 > 65535) return cudaErrorInvalidValue;
    dim3 tg(BH, (a.Nk_pad + 127) / 128);
    cudaError_t e = launch_dependent(vt_kernel, tg, dim3(256), 0, s, (const uint8_t*)a.v, (uint8_t*)a.vt, a.Nk,
                                     a.Nk_pad);
    if (e != cudaSuccess) return e;
    e = set_smem_limit_once<fwd_fp8_kernel>(F8::SMEM);
    if (e != cudaSuccess) return e;
    F8Params p;
    p.o = (__nv_bfloat16*)a.o;
    p.lse = a.lse;
    p.q_scale = a.q_scale;
    p.k_scale = a.k_scale;
    p.v_scale = a.v_scale;
    p.BH = BH;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.causal = a.causal;
    p.n_qb = (a.Nq + 127) / 128;
    p.n_kb = (a.Nk + 127) / 128;
    p.n_mtiles = (a.Nq + kFwdRowsPerCta - 1) / kFwdRowsPerCta;
    p.num_work = p.n_mtiles * BH;
    {  // heads whose K (e4m3) and V^T (e4m3), 2 Nk d bytes each, fit in 64 MiB of L2 together
        const long long per_head = 2ll * a.Nk * 128;
        const int hc_l2 = (int)std::max(1ll, std::min((long long)BH, (64ll << 20) / per_head));
        fwd_work_order(BH, a.Nq, a.Nk, a.causal, hc_l2, a.num_sms, &p.hc, &p.per_chunk);
    }
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    p.timeout_ns = a.timeout_ns;
    const int grid = p.num_work < a.num_sms ? p.num_work : a.num_sms;
    return launch_dependent(fwd_fp8_kernel, dim3(grid), dim3(F8::THREADS), F8::SMEM, s, a.map_q, a.map_k, a.map_vt, p);
}

}  // namespace fa
