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
//   bwd_dkdv  one CTA per 128-key tile (KV-tile parallel): K_j, V_j stay in
//             shared memory, Q_i / dO_i stream through a 2-stage ring;
//             tcgen05: S^T = K Q^T and dP^T = V dO^T into TMEM; S^T is read
//             out at once (so S^T of the next query tile can be issued while
//             P waits in registers); once dP^T is read, P^T and dS^T are
//             written over it as bf16 for dV += P^T dO and dK += dS^T Q, both
//             with A from TMEM; dK, dV accumulate in TMEM over all query
//             tiles.
//   bwd_dq    one CTA per 128-query tile (Q-tile parallel): Q_i, dO_i are
//             written into TMEM by the compute threads and stay; K_j / V_j
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
// HBM-bound: D/8 lanes per row, 16-byte loads, each warp with 4 row groups'
// loads in flight before it reduces.
template <int D>
constexpr int kPreRowsPerBlock = 8 * (32 / (D / 8)) * 4;

template <int D>
__global__ void __launch_bounds__(256)
bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
               float* __restrict__ delta, long long rows) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, STEPS = 4;
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
#pragma unroll 1
    for (int q4 = 0; q4 < D / 64; ++q4) {
        uint32_t v[32];
        if (!zero) {
            tmem_ld32(taddr + q4 * 32, v);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        if (valid) store_row64(dst + q4 * 32, pk, wide);
    }
}

// Shared prologue: barriers, TMEM.  Returns the TMEM base.
template <int D>
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
        tmem_alloc(smem_u32(tmem_slot), Bwd<D>::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *tmem_slot;
}

template <int D>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == Bwd<D>::MMA) {
        __syncwarp();
        tmem_dealloc(tmem, Bwd<D>::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ dK, dV (KV-tile parallel)
template <int D>
__global__ void __launch_bounds__(Bwd<D>::THREADS_DKDV, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const BwdParams p) {
    using C = Bwd<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;  // 1024-aligned (checked in bwd_setup)
    const uint32_t s_base = smem_u32(smem);
    const uint32_t bar0 = s_base + C::OFF_BAR;
    // barriers
    // S: S^T ready; SF: S^T read out of TMEM (the next S^T may overwrite it); DP: dP^T ready;
    // DS: P^T and dS^T written over dP^T (bf16, TMEM)
    // STE[s]: stage s free, once both issuers' products that read it are done (two arrivals);
    // TD, TD2: teardown of issuer 1 and 2
    const uint32_t B_KV = bar0, B_STF = bar0 + 8, B_STE = bar0 + 24, B_S = bar0 + 40, B_DP = bar0 + 48,
                   B_DS = bar0 + 56, B_ACC = bar0 + 64, B_TD = bar0 + 72, B_SF = bar0 + 80, B_TD2 = bar0 + 88;
    const uint32_t counts[12] = {1, 32, 32, 2, 2, 1, 1, 256, 1, 1, 256, 1};
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);
    const WaitCtl ctl{p.err, p.timeout_ns, abort_flag};
    const uint32_t tmem = bwd_setup<D>(smem, bar0, ctl, counts, 12);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int bh, kt;  // key tile 0 (the most query tiles when causal) first, heads in L2-sized chunks
    chunked_order(blockIdx.x, p.n_kt, p.BH, p.hc_kv, bh, kt);
    int nq, nk;
    bwd_seqlen(p, bh, nq, nk);
    const int off = nk - nq;
    int i0 = 0;
    if (p.causal) {
        const int first_q = kt * 128 - off;  // smallest query that sees key kt*128
        i0 = first_q <= 0 ? 0 : first_q / 128;
    }
    int i_end = kt * 128 < nk ? (nq + 127) / 128 : 0;  // no query tile past the sequence
    if (p.window > 0) {  // the last query that sees the tile's last key
        const long long qlast = (long long)kt * 128 + 127 - off + p.window - 1;
        i_end = qlast < 0 ? 0 : (int)min((long long)i_end, qlast / 128 + 1);
    }
    const int n = i0 < i_end ? i_end - i0 : 0;
    const uint32_t sK = s_base + C::OFF_FIXED, sV = sK + C::TILE;
    auto sQ = [&](int st) { return s_base + C::OFF_STAGE + st * 2 * C::TILE; };
    auto sDO = [&](int st) { return s_base + C::OFF_STAGE + st * 2 * C::TILE + C::TILE; };
    float* vec = (float*)(smem + C::OFF_VEC);  // stage s: lse2 at [s*256], delta at [s*256 + 128]
    const bool kv_issued = warp == C::PRODUCER && lane == 0 && n > 0 && !*abort_flag;
    if (kv_issued) {  // K and V do not come from the preprocess: they load before the wait for it
        mbar_arrive_expect_tx(B_KV, 2 * C::TILE);
        for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(sK + c * C::CHUNK, &map_k, B_KV, c * 64, kt * 128, bh, l2_policy_evict_last());
            tma_load_3d(sV + c * C::CHUNK, &map_v, B_KV, c * 64, kt * 128, bh, l2_policy_evict_last());
        }
    }
    // Launched as a programmatic dependent of the preprocess, this grid may start before D is
    // complete: every read of D comes after this wait.  Then the dQ pass launched after this grid
    // (which reads D too) may start on SMs this grid leaves free.
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
            // per-column LSE*log2(e) and D of query tile i (4 values of each per lane),
            // read from global memory one tile ahead so the load latency is off the
            // path from "stage free" to "TMA issued"
            float nl2[4], ndl[4];
            auto fetch_vec = [&](int i) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int q = i * 128 + lane + 32 * t;
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
                const int st = ii & 1, i = i0 + ii;
                if (!mbar_wait(B_STE + 8 * st, ((ii >> 1) & 1) ^ 1, ctl, kSiteBwdQEmpty)) break;
                if (lane == 0) {  // byte count first (no arrival), then the copies
                    mbar_expect_tx(B_STF + 8 * st, 2 * C::TILE);
                    for (int c = 0; c < C::KCH; ++c) {
                        tma_load_3d(sQ(st) + c * C::CHUNK, &map_q, B_STF + 8 * st, c * 64, i * 128, bh, pol);
                        tma_load_3d(sDO(st) + c * C::CHUNK, &map_do, B_STF + 8 * st, c * 64, i * 128, bh, pol);
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    vec[st * 256 + lane + 32 * t] = nl2[t];
                    vec[st * 256 + 128 + lane + 32 * t] = ndl[t];
                }
                mbar_arrive(B_STF + 8 * st);  // all 32 lanes, after their writes
                issued |= 1u << st;
                issued_par = (issued_par & ~(1u << st)) | ((uint32_t)((ii >> 1) & 1) << st);
                if (ii + 1 < n) fetch_vec(i + 1);
            }
            if (*abort_flag && lane == 0) {  // let the loads in flight land before exit
                if (kv_issued) mbar_drain(B_KV, 0, ctl, kSiteTeardown);
                for (int st = 0; st < 2; ++st)
                    if (issued & (1u << st)) mbar_drain(B_STF + 8 * st, (issued_par >> st) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA) {
        // ------------------------------------------------------------ MMA issuer 1: S^T
        // S^T(i) once S^T(i-1) has been read out of TMEM and stage i is loaded
        if (lane == 0 && !*abort_flag && n > 0) {
            bool ok = mbar_wait(B_KV, 0, ctl, kSiteBwdKvFull);
            for (int ii = 0; ii < n && ok; ++ii) {
                const int st = ii & 1;
                if (ii > 0 && !(ok = mbar_wait(B_SF, (ii - 1) & 1, ctl, kSiteBwdS))) break;
                if (!(ok = mbar_wait(B_STF + 8 * st, (ii >> 1) & 1, ctl, kSiteBwdQFull))) break;
                tc_fence_after();
                issue_ss<D>(tmem + C::COL_A, sK, sQ(st));
                mma_commit(B_S);
                mma_commit(B_STE + 8 * st);
            }
            if (*abort_flag) {
                mma_commit(B_TD);
                mbar_drain(B_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA2) {
        // ------------------------------------------------------------ MMA issuer 2: dP^T, dV, dK
        // dV(i) and dK(i) once P^T(i) and dS^T(i) are in TMEM; dP^T(i+1) over them (this
        // thread's products run in issue order, so it overwrites them only after both)
        if (lane == 0 && !*abort_flag && n > 0) {
            bool ok = mbar_wait(B_KV, 0, ctl, kSiteBwdKvFull);
            if (ok) ok = mbar_wait(B_STF, 0, ctl, kSiteBwdQFull);
            if (ok) {
                tc_fence_after();
                issue_ss<D>(tmem + C::COL_B, sV, sDO(0));
                mma_commit(B_DP);
            }
            for (int ii = 0; ii < n && ok; ++ii) {
                const int st = ii & 1;
                if (!(ok = mbar_wait(B_DS, ii & 1, ctl, kSiteBwdDS))) break;
                tc_fence_after();
                issue_ts<D>(tmem + C::COL_ACC0, tmem + C::COL_B, sDO(st), ii > 0);      // dV += P^T dO
                issue_ts<D>(tmem + C::COL_ACC1, tmem + C::COL_B + 32, sQ(st), ii > 0);  // dK += dS^T Q
                mma_commit(B_STE + 8 * st);
                if (ii + 1 < n) {
                    if (!(ok = mbar_wait(B_STF + 8 * (st ^ 1), ((ii + 1) >> 1) & 1, ctl, kSiteBwdQFull))) break;
                    tc_fence_after();
                    issue_ss<D>(tmem + C::COL_B, sV, sDO(st ^ 1));  // dP^T of the next query tile
                    mma_commit(B_DP);
                }
            }
            if (ok) mma_commit(B_ACC);
            if (*abort_flag) {
                mma_commit(B_TD2);
                mbar_drain(B_TD2, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // ------------------------------------------------------------ P^T, dS^T, epilogue
        // Two warpgroups: warpgroup h handles query columns [64h, 64h + 64) of every key row.
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // key row within the tile = TMEM lane
        const int kg = kt * 128 + r;
        const bool row_ok = kg < p.Nk;   // stored (zeros past the sequence)
        const bool key_ok = kg < nk;     // a key of the sequence
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t colA = C::COL_A + 64 * h, colB = C::COL_B + 64 * h;
        const float sc = p.scale_log2;
        bool ok = true;
        for (int ii = 0; ii < n; ++ii) {
            const int st = ii & 1, i = i0 + ii;
            const float* l2 = vec + st * 256 + 64 * h;
            const float* dl = l2 + 128;
            // key kg is visible to query q iff kg <= q + off, i.e. column c >= cmin
            const int cmin = p.causal ? kg - off - i * 128 - 64 * h : -1;
            if (!(ok = mbar_wait(B_S, ii & 1, ctl, kSiteBwdS))) break;
            tc_fence_after();
            uint32_t pp[32];
            uint32_t va[32], vb[32];
            // read this warpgroup's 64 S^T columns, then release them: the next S^T may overwrite
            tmem_ld32_async(lane_addr + colA, va);
            tmem_ld32_async(lane_addr + colA + 32, vb);
            tmem_wait_ld(va);
            tmem_wait_ld(vb);
            tc_fence_before();
            mbar_arrive(B_SF);
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
                    float a = ex2(x.x), b = ex2(x.y);
                    if constexpr (decltype(MASK)::value) {
                        if (c0 < cmin_eff || c0 > cmax_w) a = 0.f;
                        if (c0 + 1 < cmin_eff || c0 + 1 > cmax_w) b = 0.f;
                    }
                    pp[q4 * 16 + e] = pack_bf16(a, b);
                }
            }
            };
            if (__any_sync(0xffffffffu, cmin_eff > 0 || cmax_w < 63))
                p_phase(std::true_type{});
            else
                p_phase(std::false_type{});
            if (!(ok = mbar_wait(B_DP, ii & 1, ctl, kSiteBwdDP))) break;
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
                    const float a = bf_lo(pr) * (__uint_as_float(v[2 * e]) - dv[2 * e]);
                    const float b = bf_hi(pr) * (__uint_as_float(v[2 * e + 1]) - dv[2 * e + 1]);
                    pk[e] = pack_bf16(a, b);
                }
                tmem_st16_async(lane_addr + colB + 32 + q4 * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(B_DS);
        }
        if (ok) {
            bool have = n > 0;
            if (have) {
                ok = mbar_wait(B_ACC, 0, ctl, kSiteBwdDone);
                tc_fence_after();
            }
            if (ok) {
                const size_t base = ((size_t)bh * p.Nk + (row_ok ? kg : 0)) * D;
                store_acc_row<D>(lane_addr + C::COL_ACC0, p.dv + base, 1.f, row_ok, !have, h * (D / 2));
                store_acc_row<D>(lane_addr + C::COL_ACC1, p.dk + base, p.scale, row_ok, !have, h * (D / 2));
            }
        }
    }
    bwd_teardown<D>(tmem);
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
    int bh, mr;  // causal: late query tiles (most keys) first, heads in L2-sized chunks
    chunked_order(blockIdx.x, p.n_qt, p.BH, p.hc_q, bh, mr);
    const int it = p.causal ? p.n_qt - 1 - mr : mr;  // causal: late query tiles (most keys) first
    int nq, nk;
    bwd_seqlen(p, bh, nq, nk);
    const int off = nk - nq;
    int n = it * 128 < nq ? (nk + 127) / 128 : 0;  // a tile wholly past the sequence only stores zeros
    if (p.causal && n > 0) {
        const int qmax = min(it * 128 + 127, nq - 1);
        const long long lim = (long long)qmax + off;
        n = lim < 0 ? 0 : min(n, (int)(lim / 128) + 1);
    }
    int jlo = 0;  // sliding window: first key tile the tile's first query sees
    if (p.window > 0) {
        const long long lo = (long long)it * 128 + off - p.window + 1;
        jlo = lo <= 0 ? 0 : (int)min((long long)n, lo / 128);
    }
    n -= jlo;
    static_assert(NST * 2 * C::TILE <= C::OFF_VEC, "K/V stages fit below the vector region");
    auto sK = [&](int st) { return s_base + st * 2 * C::TILE; };
    auto sV = [&](int st) { return s_base + st * 2 * C::TILE + C::TILE; };

    if (warp == C::PRODUCER) {
        if (lane == 0 && !*abort_flag && n > 0) {
            const uint64_t pol = l2_policy_evict_last();
            tma_prefetch_desc(&map_k);
            tma_prefetch_desc(&map_v);
            uint32_t issued = 0, issued_par = 0;
            for (int jj = 0; jj < n; ++jj) {
                const int st = jj % NST;
                const uint32_t ph = (uint32_t)((jj / NST) & 1);
                if (!mbar_wait(B_STE + 8 * st, ph ^ 1, ctl, kSiteBwdQEmpty)) break;
                mbar_arrive_expect_tx(B_STF + 8 * st, 2 * C::TILE);
                for (int c = 0; c < C::KCH; ++c) {
                    tma_load_3d(sK(st) + c * C::CHUNK, &map_k, B_STF + 8 * st, c * 64, (jlo + jj) * 128, bh, pol);
                    tma_load_3d(sV(st) + c * C::CHUNK, &map_v, B_STF + 8 * st, c * 64, (jlo + jj) * 128, bh, pol);
                }
                issued |= 1u << st;
                issued_par = (issued_par & ~(1u << st)) | (ph << st);
            }
            if (*abort_flag) {
                for (int st = 0; st < NST; ++st)
                    if (issued & (1u << st)) mbar_drain(B_STF + 8 * st, (issued_par >> st) & 1, ctl, kSiteTeardown);
            }
        }
    } else if (warp == C::MMA) {
        if (lane == 0 && !*abort_flag && n > 0) {
            bool ok = mbar_wait(B_QA, 0, ctl, kSiteBwdQFull);
            if (ok) ok = mbar_wait(B_STF, 0, ctl, kSiteBwdKvFull);
            if (ok) {
                tc_fence_after();
                issue_ts_k<D>(tmem + C::COL_A, tmem + COL_QA, sK(0));   // S = Q K^T, Q from TMEM
                mma_commit(B_S);
                issue_ts_k<D>(tmem + C::COL_B, tmem + COL_DOA, sV(0));  // dP = dO V^T, dO from TMEM
                mma_commit(B_DP);
            }
            for (int jj = 0; jj < n && ok; ++jj) {
                const int st = jj % NST, stn = (jj + 1) % NST;
                const bool more = jj + 1 < n;
                if (more) {
                    if (!(ok = mbar_wait(B_SF, jj & 1, ctl, kSiteBwdP))) break;
                    if (!(ok = mbar_wait(B_STF + 8 * stn, ((jj + 1) / NST) & 1, ctl, kSiteBwdKvFull))) break;
                    tc_fence_after();
                    issue_ts_k<D>(tmem + C::COL_A, tmem + COL_QA, sK(stn));
                    mma_commit(B_S);
                }
                if (!(ok = mbar_wait(B_DS, jj & 1, ctl, kSiteBwdDS))) break;
                tc_fence_after();
                issue_ts<D>(tmem + C::COL_ACC0, tmem + C::COL_B, sK(st), jj > 0);  // dQ += dS K
                mma_commit(B_STE + 8 * st);
                if (more) {
                    issue_ts_k<D>(tmem + C::COL_B, tmem + COL_DOA, sV(stn));
                    mma_commit(B_DP);
                }
            }
            if (ok) mma_commit(B_ACC);
            if (*abort_flag) {
                mma_commit(B_TD);
                mbar_drain(B_TD, 0, ctl, kSiteTeardown);
            }
        }
    } else {
        // Two warpgroups: warpgroup h handles key columns [64h, 64h + 64) of every query row.
        const int h = warp >> 2;
        const int r = ((warp & 3) << 5) + lane;  // query row within the tile = TMEM lane
        const int qg = it * 128 + r;
        const bool row_ok = qg < p.Nq;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t colA = C::COL_A + 64 * h, colB = C::COL_B + 64 * h;
        float l2 = INFINITY, dl = 0.f;
        if (qg < nq) {  // a row past the sequence keeps P = 0
            const float L = p.lse[(size_t)bh * p.Nq + qg];
            l2 = (L == -INFINITY) ? INFINITY : L * kLog2e;
            dl = p.delta[(size_t)bh * p.Nq + qg];
        }
        const float sc = p.scale_log2;
        const int lim_row = p.causal ? min(qg + off, nk - 1) : nk - 1;  // last key this row sees
        // Q_i and dO_i into TMEM as the A operands of the score products: row = lane,
        // bf16 pairs in column order; warpgroup h writes d-columns [h D/2, (h+1) D/2)
        if (n > 0) {
            constexpr int W = D / 4;  // 32-bit words per half row
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const __nv_bfloat16* src = (t ? p.dO : p.q) + ((size_t)bh * p.Nq + (row_ok ? qg : 0)) * D + h * (D / 2);
                uint32_t w[W];
#pragma unroll
                for (int e = 0; e < W / 4; ++e) {
                    const uint4 x = row_ok ? __ldg(reinterpret_cast<const uint4*>(src) + e) : make_uint4(0, 0, 0, 0);
                    w[4 * e] = x.x, w[4 * e + 1] = x.y, w[4 * e + 2] = x.z, w[4 * e + 3] = x.w;
                }
                const uint32_t col = (t ? COL_DOA : COL_QA) + h * (D / 4);
                if constexpr (W == 32) {
                    tmem_st32(lane_addr + col, w);
                } else {
                    tmem_st16(lane_addr + col, w);
                }
            }
            tc_fence_before();
            mbar_arrive(B_QA);
        }
        bool ok = true;
        for (int jj = 0; jj < n; ++jj) {
            const int kb = (jlo + jj) * 128 + 64 * h;           // key of this warpgroup's column 0
            const int cmax = lim_row - kb;                       // columns > cmax are masked
            const int cmin_w = p.window > 0 ? qg + off - p.window + 1 - kb : -(1 << 30);  // and < cmin_w
            if (!(ok = mbar_wait(B_S, jj & 1, ctl, kSiteBwdS))) break;
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
                    float a = ex2(x.x), b = ex2(x.y);
                    if constexpr (decltype(MASK)::value) {
                        if (c0 > cmax || c0 < cmin_w) a = 0.f;
                        if (c0 + 1 > cmax || c0 + 1 < cmin_w) b = 0.f;
                    }
                    pp[q4 * 16 + e] = pack_bf16(a, b);
                }
            }
            };
            if (__any_sync(0xffffffffu, cmax < 63 || cmin_w > 0))
                p_phase(std::true_type{});
            else
                p_phase(std::false_type{});
            if (!(ok = mbar_wait(B_DP, jj & 1, ctl, kSiteBwdDP))) break;
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
        if (ok) {
            const bool have = n > 0;
            if (have) {
                ok = mbar_wait(B_ACC, 0, ctl, kSiteBwdDone);
                tc_fence_after();
            }
            if (ok)
                store_acc_row<D>(lane_addr + C::COL_ACC0, p.dq + ((size_t)bh * p.Nq + (row_ok ? qg : 0)) * D,
                                 p.scale, row_ok, !have, h * (D / 2));
        }
    }
    bwd_teardown<D>(tmem);
    // When launched to overlap the end of the dK/dV grid, this grid must not finish before
    // it: work that follows both on the stream may read dK and dV once this grid is done.
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
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
                                             (const __nv_bfloat16*)a.dO, a.delta, rows);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// after_pre: launched right after the preprocess on the same stream, as its
// programmatic dependent (setup and the K/V loads overlap the preprocess's end).
template <int D>
cudaError_t launch_dkdv_d(const BwdLaunch& a, cudaStream_t s, bool after_pre) {
    using C = Bwd<D>;
    static_assert(C::SMEM <= 232448, "shared memory budget");
    cudaError_t e = set_smem_limit_once<bwd_dkdv_kernel<D>>(C::SMEM);
    if (e != cudaSuccess) return e;
    const BwdParams p = make_params(a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_kt * p.BH));
    cfg.blockDim = dim3(C::THREADS_DKDV);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_pre ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<D>, a.map_q, a.map_k, a.map_v, a.map_do, p);
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
    cfg.gridDim = dim3((unsigned)(p.n_qt * p.BH));
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

}  // namespace

cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_pre_d<128>(a, s) : launch_pre_d<64>(a, s);
}
cudaError_t launch_bwd_dkdv(const BwdLaunch& a, cudaStream_t s, bool after_pre) {
    return a.d == 128 ? launch_dkdv_d<128>(a, s, after_pre) : launch_dkdv_d<64>(a, s, after_pre);
}
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t s, bool after_dkdv) {
    return a.d == 128 ? launch_dq_d<128>(a, s, after_dkdv) : launch_dq_d<64>(a, s, after_dkdv);
}

}  // namespace fa
