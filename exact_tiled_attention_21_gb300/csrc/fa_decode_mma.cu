// Paged, grouped-query decode on the tensor cores (d = 128).
//
// Same result as the split-KV decode (fa_decode.cu): per split of a
// sequence's keys, a partial output and a partial log-sum-exp, merged by the
// LSE-weighted combine (wiki.ai-engineering.at "Flash Attention", "Lösung:
// Online Softmax").  The cache is paged (johe.ru "Flash Attention: ...",
// "Альтернативы": PagedAttention) and the query heads of one kv head share it,
// so one pass over a kv head's pages serves its whole group of query heads:
// the group's q rows against the keys is a small dense product, done here on
// the tensor cores with the keys as the 128-row M side.
//
// GB300 mapping (one persistent CTA per SM, 224 threads, 64 TMEM columns).
// Work item = (sequence b, kv head, group of up to 16 query heads, split s):
// keys [k0, k1) of sequence b, in stages of 128 keys.
//   warp 4      TMA producer of K: the group's 16 q rows (rows past the group
//               are other heads or zero fill; their columns are never used),
//               then per stage the K rows of the pages the stage covers (block
//               table read 32 entries at a time, two work items ahead), in
//               boxes of R = gcd(page, 128) rows, so a box never crosses a
//               page (a page of 48 tokens is three boxes of 16), two per box
//               position (one per 64-feature half: the score product needs
//               all 128 keys of a half at one row stride), or one holding
//               both halves when d = 128 and the boxes have 8 rows.
//   warp 6      TMA producer of V: one box per R rows holding both halves
//               (the value product steps through the keys 16 at a time and
//               takes each step's address on its own).  A page index outside
//               the pool is loaded from an out-of-range coordinate, which the
//               TMA fills with zeros.
//   warp 5      MMA issuer: S^T = K Q^T (M = 128 keys, N = 16 heads, K = d)
//               into TMEM, and O^T += V^T P^T (M = d, N = 16, K = 128 keys),
//               V read MN-major from the slot it was loaded into.
//   warps 0-3   thread = key of the stage: per-head maximum of the scores over
//               the 128 keys (butterfly across the warp, named barrier across
//               warps), p = 2^(s c - m) written as bf16 P^T into shared memory
//               (K-major, 128-byte swizzle), per-thread partial sums reduced
//               once per item.  Thread = feature row of O^T for the lazy
//               rescale (only when a head's maximum grew by more than 2^8) and
//               for the epilogue: partial o / l and lse = (m + log2 l) ln 2.
//   Keys of the last stage at or past k1 get p = 0 and their V rows are
//   zeroed in shared memory before the product (the unused tail of a page may
//   hold anything, and 0 * NaN would not vanish).
#include <algorithm>

#include "fa_internal.h"

namespace fa {
namespace {

template <int D_>
struct Dm {
    static constexpr int D = D_;                  // 128 or 64
    static constexpr int BK = 128;                // keys per stage
    static constexpr int NG = 16;                 // query heads per work item (MMA N of the scores)
    static constexpr int SLOT = BK * D * 2;       // one K or V stage: 32 KB (d = 128), 16 KB (d = 64)
    static constexpr int CHUNK = BK * 128;        // 64 features x 128 keys (the two halves of d = 128)
    static constexpr int NSLOT = D == 128 ? 3 : 6;  // stages in flight, K and V rings each (192 KB either way)
    static constexpr int Q_BYTES = NG * D * 2;
    static constexpr int QCHUNK = NG * 128;       // 64 features x 16 rows
    static constexpr int P_BYTES = NG * BK * 2;   // 4 KB
    static constexpr int PCHUNK = NG * 128;       // 64 keys x 16 heads
    static constexpr int OFF_K = 0;               // K ring: [feature half][128 keys][128 B] per slot
    static constexpr int OFF_V = NSLOT * SLOT;    // V ring: pages back to back, [half][page rows][128 B] each
    static constexpr int OFF_Q = 2 * NSLOT * SLOT;  // 2 buffers
    static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;  // 2 buffers
    static constexpr int OFF_RED = OFF_P + 2 * P_BYTES;  // fp32 max [2][4][16], sums [4][16]
    static constexpr int OFF_X = OFF_RED + (2 * 4 * 16 + 4 * 16) * 4;  // d = 64: the second O^T half, [64][16] fp32
    static constexpr int OFF_LENS = OFF_X + (D == 64 ? 64 * 16 * 4 : 0);  // int32 [MAX_B]
    static constexpr int MAX_B = 2048;  // lengths staged in shared memory (later ones read from global)
    static constexpr int OFF_BAR = OFF_LENS + MAX_B * 4;
    // k_full, k_empty, v_full, v_empty [NSLOT each], q_full[2], q_empty[2], s_full[2], p_ready[2], pv_done[2],
    // o_final, teardown
    static constexpr int NBAR = 4 * NSLOT + 12;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static constexpr int THREADS = 224;
    static constexpr uint32_t TMEM_COLS = 64;
    static constexpr uint32_t COL_S = 0;          // two 16-column S^T buffers
    static constexpr uint32_t COL_O = 32;         // O^T: 16 columns (d = 128) or 32 (d = 64, below)
    // d = 64: the value product runs with M = 128 rows = (64 features) x (keys 0-63 | keys 64-127)
    // and N = 32 columns = (16 heads) x (the same two key halves); only the two diagonal blocks
    // are used, and O^T[f][h] = D[f][h] + D[64 + f][16 + h]
    static constexpr int NO = D == 128 ? NG : 2 * NG;
    static constexpr uint32_t IDESC_S = idesc_bf16(128, NG, 0, 0);  // K, Q both K-major
    static constexpr uint32_t IDESC_O = idesc_bf16(128, NO, 1, 0);  // V^T MN-major, P^T K-major
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "operand tiles need 1024-byte alignment");
};

struct MmaParams {
    const int* table;  // null: the identity table (page b * max_pages + i) of a contiguous cache
    const int* lens;   // null: every sequence is max_pages * page long
    float* part_o;
    float* part_lse;
    int B, Hq, Hkv, g, page, max_pages, num_pages, splits, ngrp, nitems;
    float scale_log2;
    DevError* err;
    uint64_t timeout_ns;
};

struct Item {
    int b, kvh, h0, gcount, split, k0, k1;
};

// Work item w -> (sequence, kv head, head group of NH, split) and its keys:
// ceil(len / splits) rounded up to whole 128-key stages per split.  32-bit
// unsigned arithmetic: len < 2^31 and splits <= 256 keep every term in range.
template <int NH>
__device__ __forceinline__ Item item_at(const MmaParams& p, int w, int len) {
    Item it;
    unsigned t = (unsigned)w;
    it.split = (int)(t % (unsigned)p.splits);
    t /= (unsigned)p.splits;
    const int grp = (int)(t % (unsigned)p.ngrp);
    t /= (unsigned)p.ngrp;
    it.kvh = (int)(t % (unsigned)p.Hkv);
    it.b = (int)(t / (unsigned)p.Hkv);
    it.h0 = it.kvh * p.g + grp * NH;
    it.gcount = min(NH, p.g - grp * NH);
    const unsigned chunk = (((unsigned)len + (unsigned)p.splits - 1u) / (unsigned)p.splits + 127u) & ~127u;
    const unsigned k0 = chunk * (unsigned)it.split;
    it.k0 = (int)min(k0, (unsigned)len);
    it.k1 = (int)min(k0 + chunk, (unsigned)len);
    return it;
}

// Rows per TMA box of a page: gcd(page, 128), i.e. the lowest set bit of the page size capped at
// 128 (page sizes are multiples of 8).  Stages start at multiples of 128 keys, so a box of R rows
// at key key0 + i R starts at a multiple of R within one page and ends inside it.
__device__ __forceinline__ int box_rows(int page) { return min(page & -page, 128); }

// A length outside [1, max_pages * page] is out of range: clamped, never
// dereferenced past the table (recorded when the lengths are staged).
__device__ __forceinline__ int clamp_len(const MmaParams& p, int len) {
    const int cap = p.max_pages * p.page;
    return len < 1 ? 0 : min(len, cap);
}

// Length of sequence b: staged in shared memory for the first MAX_B sequences, read (and clamped)
// from global memory past them.
template <int D>
__device__ __forceinline__ int seq_len(const MmaParams& p, int b, const int* s_lens) {
    if (b < Dm<D>::MAX_B) return s_lens[b];
    return clamp_len(p, p.lens ? __ldg(p.lens + b) : p.max_pages * p.page);
}

template <int D, int NH>
__device__ __forceinline__ Item item_of(const MmaParams& p, int w, const int* s_lens) {
    const int b = (int)((unsigned)w / ((unsigned)p.splits * p.ngrp * p.Hkv));
    return item_at<NH>(p, w, seq_len<D>(p, b, s_lens));
}

// Butterfly over the 32 lanes of a warp for NH values per lane (NH = 4, 8,
// 16): each level sends half of what a lane holds to its partner and keeps the
// other half, until one value is left, then the remaining levels reduce it
// fully.  Returns, in lane l, the reduction over the warp of value l / (32 / NH).
template <bool MAX, int NH>
__device__ __forceinline__ float bfly(const float (&v)[NH], int lane) {
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
    float cur[NH];
#pragma unroll
    for (int i = 0; i < NH; ++i) cur[i] = v[i];
#pragma unroll
    for (int n = NH / 2, m = 16; n >= 1; n >>= 1, m >>= 1) {
        const bool hi = lane & m;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = hi ? cur[i] : cur[i + n], keep = hi ? cur[i + n] : cur[i];
            cur[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, m));
        }
    }
    float d = cur[0];
#pragma unroll
    for (int m = 16 / NH; m >= 1; m >>= 1) d = op(d, __shfl_xor_sync(0xffffffffu, d, m));
    return d;
}

template <int D, int NH>
__global__ void __launch_bounds__(Dm<D>::THREADS, 1)
decode_paged_mma_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const MmaParams p) {
    static_assert(NH == 4 || NH == 8 || NH == 16, "heads per item");
    using Dm = fa::Dm<D>;
    constexpr int LPH = 32 / NH;  // lanes per head after the butterfly
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + Dm::OFF_BAR;
    // ring barriers of stage g: slot g % NSLOT; kv = 0 for K, 1 for V
    auto bar_full = [&](int kv, uint32_t g) { return bar0 + 8 * (kv * 2 * Dm::NSLOT + g % Dm::NSLOT); };
    auto bar_empty = [&](int kv, uint32_t g) { return bar0 + 8 * (kv * 2 * Dm::NSLOT + Dm::NSLOT + g % Dm::NSLOT); };
    auto ring_par = [](uint32_t g) { return (g / Dm::NSLOT) & 1; };
    const uint32_t BAR_QF = bar0 + 32 * Dm::NSLOT;  // + 8 * buffer
    const uint32_t BAR_QE = BAR_QF + 16;
    const uint32_t BAR_SF = BAR_QE + 16;
    const uint32_t BAR_PR = BAR_SF + 16;
    const uint32_t BAR_PV = BAR_PR + 16;
    const uint32_t BAR_OF = BAR_PV + 16;
    const uint32_t BAR_TD = BAR_OF + 8;
    uint32_t* tmem_slot = (uint32_t*)(smem + Dm::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + Dm::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < 4 * Dm::NSLOT; ++s) mbar_init(bar0 + 8 * s, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR_QF + 8 * i, 1);
            mbar_init(BAR_QE + 8 * i, 1);
            mbar_init(BAR_SF + 8 * i, 1);
            mbar_init(BAR_PR + 8 * i, 128);
            mbar_init(BAR_PV + 8 * i, 1);
        }
        mbar_init(BAR_OF, 1);
        mbar_init(BAR_TD, 1);
        fence_mbar_init();
        if ((s_base & 1023u) != 0) record_error(ctl, kErrTimeout, kSiteAlign, (int)(s_base & 1023u));
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), Dm::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_launch_dependents();
    pdl_wait();  // the setup above may overlap the kernel before; its writes are visible from here
    // sequence lengths, clamped to the table (every role reads them per item)
    int* s_lens = reinterpret_cast<int*>(smem + Dm::OFF_LENS);
    for (int b = tid; b < p.B; b += Dm::THREADS) {
        const int raw = p.lens ? __ldg(p.lens + b) : p.max_pages * p.page;
        const int len = clamp_len(p, raw);
        if (b < Dm::MAX_B) s_lens[b] = len;
        if (len != raw && blockIdx.x == 0 && atomicCAS(&p.err->code, 0, kErrInvalid) == 0) {
            p.err->site = kSitePagedTable;
            p.err->block = b;
            p.err->aux = raw;
        }
    }
    if (NH < Dm::NG && tid < 128) {  // P^T rows of the unused MMA columns stay zero
        uint4* pz = reinterpret_cast<uint4*>(smem + Dm::OFF_P);
        for (int i = tid; i < 2 * Dm::P_BYTES / 16; i += 128) {
            const int row = (i * 16 % Dm::PCHUNK) / 128;
            if (row >= NH) pz[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int first = blockIdx.x;
    const int grid = gridDim.x;

    if (warp == 4 || warp == 6) {
        // ------------------------------------------------------------ TMA producers (whole warps)
        const int kv = warp == 6;  // 0: q and K, 1: V
        const uint64_t pol_q = l2_policy_evict_last();
        const uint64_t pol_kv = l2_policy_evict_first();
        if (lane == 0) {
            if (!kv) tma_prefetch_desc(&map_q);
            tma_prefetch_desc(kv ? &map_v : &map_k);
        }
        uint32_t g = 0, qn = 0, issued = 0, issued_par = 0;
        bool ok = !*abort_flag;
        // Block-table entries (lane i: page k0/page + i of an item) are loaded
        // two items ahead, so their latency hides behind two items of copies.
        auto first_entries = [&](int w2) {
            if (w2 >= p.nitems) return 0;
            const Item n = item_of<D, NH>(p, w2, s_lens);
            const int pi = n.k0 / p.page + lane;
            if (!(n.k0 < n.k1 && pi < p.max_pages)) return 0;
            return p.table ? __ldg(p.table + (size_t)n.b * p.max_pages + pi) : n.b * p.max_pages + pi;
        };
        int tb0 = first_entries(first), tb1 = first_entries(first + grid);
        for (int w = first; w < p.nitems && ok; w += grid) {
            const Item it = item_of<D, NH>(p, w, s_lens);
            int tbl = tb0;
            tb0 = tb1;
            tb1 = first_entries(w + 2 * grid);
            if (it.k0 >= it.k1) continue;
            if (!kv) {
                const uint32_t qb = qn & 1;
                if (lane == 0) {
                    if (qn >= 2) ok = mbar_wait(BAR_QE + 8 * qb, ((qn >> 1) - 1) & 1, ctl, kSitePagedQ);
                    if (ok) {
                        mbar_arrive_expect_tx(BAR_QF + 8 * qb, Dm::Q_BYTES);
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_3d(s_base + Dm::OFF_Q + qb * Dm::Q_BYTES + c * Dm::QCHUNK, &map_q,
                                        BAR_QF + 8 * qb, c * 64, it.b * p.Hq + it.h0, 0, pol_q);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++qn;
            }
            const int* trow = p.table ? p.table + (size_t)it.b * p.max_pages : nullptr;
            const int rows = box_rows(p.page);
            int tbl_base = it.k0 / p.page;  // tbl (lane i) = entry of page tbl_base + i
            for (int key0 = it.k0; key0 < it.k1; key0 += Dm::BK, ++g) {
                const int nk = min(Dm::BK, it.k1 - key0);
                const int nbox = (nk + rows - 1) / rows;  // lane i < nbox: rows key0 + i R ..
                const int pfirst = key0 / p.page, plast = (key0 + (nbox - 1) * rows) / p.page;
                const int key = key0 + min(lane, nbox - 1) * rows;  // below k1: no overflow
                const int pidx = key / p.page;       // this lane's page (lanes < nbox)
                const int prow = key - pidx * p.page;  // its first row there: a multiple of R
                if (plast >= tbl_base + 32) {  // at most 17 pages per stage (R >= 8)
                    tbl_base = pfirst;
                    const int pi = pfirst + lane;
                    tbl = pi < p.max_pages ? (trow ? __ldg(trow + pi) : it.b * p.max_pages + pi) : 0;
                }
                int pg = __shfl_sync(0xffffffffu, tbl, (pidx - tbl_base) & 31);
                if (lane < nbox && (pg < 0 || pg >= p.num_pages)) {
                    if (atomicCAS(&p.err->code, 0, kErrInvalid) == 0) {
                        p.err->site = kSitePagedTable;
                        p.err->block = blockIdx.x;
                        p.err->aux = pg;
                    }
                    pg = p.num_pages;  // wholly out of range: zero fill
                }
                if (lane == 0) {
                    ok = mbar_wait(bar_empty(kv, g), ring_par(g) ^ 1, ctl, kSitePagedKv);
                    if (ok) mbar_arrive_expect_tx(bar_full(kv, g), (uint32_t)(nbox * rows * D * 2));
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane < nbox) {
                    if (!kv && D == 128 && rows == 8) {
                        // 8-row boxes: both feature halves in one box, [half][8 rows][128 B] (the score
                        // product then steps 2 KB per 8 keys and 1 KB to the second half)
                        const uint32_t dst = s_base + Dm::OFF_K + (g % Dm::NSLOT) * Dm::SLOT + (uint32_t)(lane * rows * 256);
                        tma_load_5d(dst, &map_k, bar_full(0, g), 0, prow, 0, it.kvh, pg, pol_kv);
                    } else if (!kv) {
                        const uint32_t dst = s_base + Dm::OFF_K + (g % Dm::NSLOT) * Dm::SLOT + (uint32_t)(lane * rows * 128);
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(dst + c * Dm::CHUNK, &map_k, bar_full(0, g), c * 64, prow, it.kvh, pg, pol_kv);
                    } else if constexpr (D == 128) {
                        const uint32_t dst = s_base + Dm::OFF_V + (g % Dm::NSLOT) * Dm::SLOT + (uint32_t)(lane * rows * 256);
                        tma_load_5d(dst, &map_v, bar_full(1, g), 0, prow, 0, it.kvh, pg, pol_kv);
                    } else {  // d = 64: a box's rows are whole 128-byte rows, back to back
                        const uint32_t dst = s_base + Dm::OFF_V + (g % Dm::NSLOT) * Dm::SLOT + (uint32_t)(lane * rows * 128);
                        tma_load_4d(dst, &map_v, bar_full(1, g), 0, prow, it.kvh, pg, pol_kv);
                    }
                }
                issued |= 1u << (g % Dm::NSLOT);
                issued_par = (issued_par & ~(1u << (g % Dm::NSLOT))) | (ring_par(g) << (g % Dm::NSLOT));
            }
        }
        if (lane == 0 && *abort_flag) {  // let every load in flight land before the CTA exits
            if (!kv)
                for (uint32_t i = (qn >= 2 ? qn - 2 : 0); i < qn; ++i)
                    mbar_drain(BAR_QF + 8 * (i & 1), (i >> 1) & 1, ctl, kSiteTeardown);
            for (uint32_t s2 = 0; s2 < (uint32_t)Dm::NSLOT; ++s2)
                if (issued & (1u << s2)) mbar_drain(bar_full(kv, s2), (issued_par >> s2) & 1, ctl, kSiteTeardown);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        // Stage g uses fills 2g (K) and 2g + 1 (V).  The scores S_g and the
        // product PV_g are issued as soon as their inputs are ready, S at most
        // one stage ahead of PV (two S^T buffers), each in stage order.
        if (lane == 0 && !*abort_flag) {
            // V^T operand: each 16-key step starts at its own address (boxes of
            // R = gcd(page, 128) rows, [half][R rows][128 B] each, back to back)
            const int R = box_rows(p.page);
            const uint32_t v_lbo = (uint32_t)R * 128, v_sbo = R == 8 ? 2048u : 1024u;
            // K operand: [half][128 keys][128 B], or at d = 128 with 8-row boxes [box][half][8 rows][128 B]
            const bool k_boxed = D == 128 && R == 8;
            const uint32_t k_half = k_boxed ? 1024u : (uint32_t)Dm::CHUNK, k_sbo = k_boxed ? 2048u : 1024u;
            uint32_t v_off[Dm::BK / 16];
#pragma unroll
            for (int k = 0; k < Dm::BK / 16; ++k) v_off[k] = (uint32_t)((16 * k) / R * (R * 256) + (16 * k) % R * 128);
            struct Cur {
                int w, j, nst;
                uint32_t g, q;  // global stage, item ordinal (Q buffer use)
            };
            auto seek = [&](Cur& c, int w) {  // first item with keys at or after w
                for (; w < p.nitems; w += grid) {
                    const Item it = item_of<D, NH>(p, w, s_lens);
                    if (it.k0 < it.k1) {
                        c.w = w;
                        c.j = 0;
                        c.nst = (it.k1 - it.k0 + Dm::BK - 1) / Dm::BK;
                        return;
                    }
                }
                c.w = p.nitems;
            };
            Cur cs{0, 0, 0, 0u, 0u}, cv{0, 0, 0, 0u, 0u};
            seek(cs, first);
            seek(cv, first);
            uint64_t t_idle = 0;
            uint32_t spins = 0;
            while (cv.w < p.nitems) {
                bool prog = false;
                if (cs.w < p.nitems && cs.g <= cv.g + 1) {
                    const uint32_t qb = cs.q & 1;
                    if ((cs.j > 0 || mbar_test(BAR_QF + 8 * qb, (cs.q >> 1) & 1)) &&
                        mbar_test(bar_full(0, cs.g), ring_par(cs.g))) {
                        tc_fence_after();
                        const uint32_t sQ = s_base + Dm::OFF_Q + qb * Dm::Q_BYTES;
                        const uint32_t sK = s_base + Dm::OFF_K + (cs.g % Dm::NSLOT) * Dm::SLOT;
#pragma unroll
                        for (int k = 0; k < Dm::D / 16; ++k)
                            mma_ss(tmem + Dm::COL_S + (cs.g & 1) * Dm::NG,
                                   sdesc_sw128(sK + (k >> 2) * k_half + (k & 3) * 32, 16, k_sbo),
                                   sdesc_sw128(sQ + (k >> 2) * Dm::QCHUNK + (k & 3) * 32, 16, 1024), Dm::IDESC_S,
                                   k > 0);
                        mma_commit(BAR_SF + 8 * (cs.g & 1));
                        mma_commit(bar_empty(0, cs.g));
                        if (++cs.j == cs.nst) {
                            mma_commit(BAR_QE + 8 * qb);
                            ++cs.q;
                            seek(cs, cs.w + grid);
                        }
                        ++cs.g;
                        prog = true;
                    }
                }
                if (cv.g < cs.g) {
                    if (mbar_test(BAR_PR + 8 * (cv.g & 1), (cv.g >> 1) & 1) && mbar_test(bar_full(1, cv.g), ring_par(cv.g))) {
                        tc_fence_after();
                        const uint32_t sV = s_base + Dm::OFF_V + (cv.g % Dm::NSLOT) * Dm::SLOT;
                        const uint32_t sP = s_base + Dm::OFF_P + (cv.g & 1) * Dm::P_BYTES;
                        if constexpr (D == 128) {
#pragma unroll
                            for (int k = 0; k < Dm::BK / 16; ++k)
                                mma_ss(tmem + Dm::COL_O, sdesc_sw128(sV + v_off[k], v_lbo, v_sbo),
                                       sdesc_sw128(sP + (k >> 2) * Dm::PCHUNK + (k & 3) * 32, 16, 1024), Dm::IDESC_O,
                                       (cv.j > 0 || k > 0) ? 1u : 0u);
                        } else {
                            // M-block 0: keys 16k.. (rows of 128 B), M-block 1: keys 64 + 16k.. (LBO
                            // 8 KB); B: 32 rows = both 64-key chunks of P^T, contiguous
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_ss(tmem + Dm::COL_O, sdesc_sw128(sV + 2048 * k, 64 * 128, 1024),
                                       sdesc_sw128(sP + 32 * k, 16, 1024), Dm::IDESC_O, (cv.j > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(BAR_PV + 8 * (cv.g & 1));
                        mma_commit(bar_empty(1, cv.g));
                        if (++cv.j == cv.nst) {
                            mma_commit(BAR_OF);
                            seek(cv, cv.w + grid);
                        }
                        ++cv.g;
                        prog = true;
                    }
                }
                if (prog) {
                    spins = 0;
                } else if ((++spins & 63u) == 0) {
                    if (*abort_flag) break;
                    const uint64_t now = globaltimer();
                    if (spins == 64) {
                        t_idle = now;
                    } else if (now - t_idle > p.timeout_ns) {
                        record_error(ctl, kErrTimeout, kSitePagedP, (int)cv.g);
                        break;
                    }
                }
            }
            if (*abort_flag) {  // every MMA issued so far must finish before TMEM is freed
                mma_commit(BAR_TD);
                mbar_drain(BAR_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue (warps 0-3)
        const int r = tid;  // key of the stage (row of S^T) and feature row of O^T
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        float* red_m = reinterpret_cast<float*>(smem + Dm::OFF_RED);  // [2][4][16]
        float* red_l = red_m + 2 * 4 * 16;                             // [4][16]
        const float c = p.scale_log2;
        uint32_t gs = 0, items = 0;
        const int R = box_rows(p.page);
        bool failed = false;
        for (int w = first; w < p.nitems && !failed; w += grid) {
            const Item it = item_of<D, NH>(p, w, s_lens);
            const size_t head0 = (size_t)it.b * p.Hq + it.h0;
            if (it.k0 >= it.k1) {  // empty split: weight 0 in the combine
                if (r < D)
                    for (int h = 0; h < it.gcount; ++h)
                        p.part_o[((size_t)(head0 + h) * p.splits + it.split) * Dm::D + r] = 0.f;
                if (r < it.gcount) p.part_lse[(size_t)(head0 + r) * p.splits + it.split] = -INFINITY;
                continue;
            }
            const int nst = (it.k1 - it.k0 + Dm::BK - 1) / Dm::BK;
            float m_run[NH], lp[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) m_run[h] = -INFINITY, lp[h] = 0.f;
            bool ok = true;
            for (int j = 0; j < nst; ++j, ++gs) {
                const int nk = min(Dm::BK, it.k1 - it.k0 - j * Dm::BK);
                const bool valid = r < nk;
                const uint32_t sb = gs & 1;
                if (ok) ok = mbar_wait(BAR_SF + 8 * sb, (gs >> 1) & 1, ctl, kSitePagedS);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                uint32_t sv[16];
                if (ok) {
                    tmem_ld16(lane_addr + Dm::COL_S + sb * Dm::NG, sv);
                } else {
#pragma unroll
                    for (int h = 0; h < 16; ++h) sv[h] = 0u;
                }
                float x[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) x[h] = valid ? __uint_as_float(sv[h]) : -INFINITY;
                const float mh = bfly<true, NH>(x, lane);
                if (lane % LPH == 0) red_m[(sb * 4 + warp) * 16 + lane / LPH] = mh;
                if (!bar_and(1, 128, ok)) {
                    failed = true;
                    break;
                }
                float m_new[NH];
                bool grow = false;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const float* rm = red_m + sb * 64 + h;
                    const float mx = fmaxf(fmaxf(rm[0], rm[16]), fmaxf(rm[32], rm[48]));
                    m_new[h] = fmaxf(m_run[h], mx * c);
                    grow |= m_new[h] > m_run[h] + 8.f;
                }
                if (j == 0) {
#pragma unroll
                    for (int h = 0; h < NH; ++h) m_run[h] = m_new[h];
                } else if (grow) {  // the same decision in every thread: rescale O^T and the sums
                    float alpha[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h) alpha[h] = (m_new[h] == -INFINITY) ? 1.f : ex2(m_run[h] - m_new[h]);
                    if (ok) ok = mbar_wait(BAR_PV + 8 * ((gs - 1) & 1), ((gs - 1) >> 1) & 1, ctl, kSitePagedPv);
                    ok = __all_sync(0xffffffffu, ok);
                    tc_fence_after();
                    if (ok) {
                        if constexpr (D == 128) {
                            uint32_t ov[16];
                            tmem_ld16(lane_addr + Dm::COL_O, ov);
#pragma unroll
                            for (int h = 0; h < NH; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                            tmem_st16(lane_addr + Dm::COL_O, ov);
                        } else {  // both key halves of every head
                            uint32_t ov[32];
                            tmem_ld32(lane_addr + Dm::COL_O, ov);
#pragma unroll
                            for (int h = 0; h < NH; ++h) {
                                ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                                ov[16 + h] = __float_as_uint(__uint_as_float(ov[16 + h]) * alpha[h]);
                            }
                            tmem_st32(lane_addr + Dm::COL_O, ov);
                        }
                    }
#pragma unroll
                    for (int h = 0; h < NH; ++h) lp[h] *= alpha[h], m_run[h] = m_new[h];
                }
                // P^T buffer sb is free once the product of stage gs - 2 is done
                if (gs >= 2 && ok) ok = mbar_wait(BAR_PV + 8 * sb, ((gs >> 1) - 1) & 1, ctl, kSitePagedPv);
                {
                    uint8_t* pbuf = smem + Dm::OFF_P + sb * Dm::P_BYTES + (r >> 6) * Dm::PCHUNK + (r & 7) * 2;
                    const int u = (r & 63) >> 3;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const float pv = ex2(fmaf(x[h], c, -m_run[h]));
                        lp[h] += pv;
                        *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + ((u ^ (h & 7)) << 4)) = __float2bfloat16_rn(pv);
                    }
                }
                if (nk < Dm::BK) {  // last stage: zero the V rows of keys past the split
                    if (ok) ok = mbar_wait(bar_full(1, gs), ring_par(gs), ctl, kSitePagedKv);
                    if (!valid) {
                        uint4* row = reinterpret_cast<uint4*>(smem + Dm::OFF_V + (gs % Dm::NSLOT) * Dm::SLOT +
                                                              (r / R) * (R * 2 * D) + (r % R) * 128);
                        const int half = R * 128 / 16;  // uint4s from a row of one half to the other
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            row[i] = make_uint4(0u, 0u, 0u, 0u);
                            if (D == 128) row[half + i] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                mbar_arrive(BAR_PR + 8 * sb);
            }
            if (failed) break;
            // ---------------- epilogue: partial o / l and lse of the group's heads
            const float lh = bfly<false, NH>(lp, lane);
            if (lane % LPH == 0) red_l[warp * 16 + lane / LPH] = lh;
            if (!bar_and(1, 128, ok)) {
                failed = true;
                break;
            }
            float inv_l[NH];
            float lse = -INFINITY;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float l = (red_l[h] + red_l[16 + h]) + (red_l[32 + h] + red_l[48 + h]);
                inv_l[h] = __frcp_rn(l);
                if (h == r) lse = (m_run[h] + lg2(l)) * 0.69314718055994531f;
            }
            if (ok) ok = mbar_wait(BAR_OF, items & 1, ctl, kSitePagedO);
            ++items;
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            float* po = p.part_o + ((size_t)head0 * p.splits + it.split) * Dm::D + r;
            if constexpr (D == 128) {
                uint32_t ov[16];
                if (ok) {
                    tmem_ld16(lane_addr + Dm::COL_O, ov);
                } else {
#pragma unroll
                    for (int h = 0; h < 16; ++h) ov[h] = 0u;
                }
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    if (h < it.gcount) po[(size_t)h * p.splits * Dm::D] = __uint_as_float(ov[h]) * inv_l[h];
            } else {
                // feature r < 64: its keys 0-63 part in its own lane (columns h), its keys 64-127
                // part in lane 64 + r (columns 16 + h), handed over through shared memory
                uint32_t ov[32];
                if (ok) {
                    tmem_ld32(lane_addr + Dm::COL_O, ov);
                } else {
#pragma unroll
                    for (int h = 0; h < 32; ++h) ov[h] = 0u;
                }
                float* xo = reinterpret_cast<float*>(smem + Dm::OFF_X);
                if (r >= 64) {
#pragma unroll
                    for (int h = 0; h < NH; ++h) xo[(r - 64) * 16 + ((h + r) & 15)] = __uint_as_float(ov[16 + h]);
                }
                if (!bar_and(1, 128, ok)) {
                    failed = true;
                    break;
                }
                if (r < 64) {
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        if (h < it.gcount)
                            po[(size_t)h * p.splits * Dm::D] =
                                (__uint_as_float(ov[h]) + xo[r * 16 + ((h + r) & 15)]) * inv_l[h];
                }
            }
            if (r < it.gcount) p.part_lse[(size_t)(head0 + r) * p.splits + it.split] = lse;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) {
        __syncwarp();
        tmem_dealloc(tmem, Dm::TMEM_COLS);
    }
}

template <int D, int NH>
cudaError_t launch_nh(const PagedDecodeLaunch& a, MmaParams p, cudaStream_t s) {
    using C = Dm<D>;
    p.ngrp = (p.g + NH - 1) / NH;
    const long long nitems = (long long)a.B * a.Hkv * p.ngrp * a.splits;
    if (nitems > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    p.nitems = (int)nitems;
    cudaError_t e = set_smem_limit_once<decode_paged_mma_kernel<D, NH>>(C::SMEM);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<long long>(nitems, a.num_sms);
    return launch_dependent(decode_paged_mma_kernel<D, NH>, dim3(grid), dim3(C::THREADS), C::SMEM, s, a.map_q,
                            a.map_k, a.map_v, p);
}

template <int D>
cudaError_t launch_d(const PagedDecodeLaunch& a, const MmaParams& p, cudaStream_t s) {
    // heads per work item: the group, in MMA columns of 4, 8 or 16
    return p.g <= 4 ? launch_nh<D, 4>(a, p, s) : p.g <= 8 ? launch_nh<D, 8>(a, p, s) : launch_nh<D, 16>(a, p, s);
}

}  // namespace

cudaError_t launch_decode_paged_mma(const PagedDecodeLaunch& a, cudaStream_t s) {
    if (a.d != 64 && a.d != 128) return cudaErrorInvalidValue;
    MmaParams p;
    p.B = a.B;
    p.table = a.table;
    p.lens = a.lens;
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.g = a.Hq / a.Hkv;
    p.page = a.page;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.splits = a.splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    p.timeout_ns = a.timeout_ns;
    cudaError_t e = a.d == 128 ? launch_d<128>(a, p, s) : launch_d<64>(a, p, s);
    if (e != cudaSuccess) return e;
    return launch_decode_combine(a.part_o, a.part_lse, a.o, a.lse, a.B * a.Hq, a.splits, a.d, s);
}

}  // namespace fa
