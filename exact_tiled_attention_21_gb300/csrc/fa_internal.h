// Internal launch interfaces between the C-ABI layer (fa_api.cu) and the
// kernel translation units.  Arguments arrive here already validated.
#pragma once

#include <atomic>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_ptx.cuh"

namespace fa {

// Item sequence of persistent CTA c (of G) over n_items work items listed in
// chunks of chunk_items (heads whose streamed operands fit in L2 together).
// per_chunk (items of unequal weight, heaviest first within each chunk): the
// CTAs take each chunk round by round, alternating direction (round r:
// r*G + c, or r*G + G-1-c), and odd chunks start reversed, so that the
// rounds' long and short items even out per CTA while the CTAs in flight stay
// within one chunk.  Otherwise (equal weights), and with chunks smaller than
// the grid, the rounds run over the whole list, which keeps every CTA's count
// within one item (and with the list heaviest first, CTA 0 takes the heaviest
// item of one round and the lightest of the next).  Returns n_items once the
// CTA has no more.  Host and device (the host replays the schedule to size
// grids).
struct ItemSeq {
    int ci = 0, rd = 0;  // chunk, and round within it
};
__host__ __device__ inline int next_chunked_item(ItemSeq& q, int n_items, int chunk_items, int G, int c,
                                                 bool per_chunk) {
    if (!per_chunk || chunk_items < G) {
        const int rd = q.rd++;
        const int w = rd * G + ((rd & 1) ? G - 1 - c : c);
        return w < n_items ? w : n_items;
    }
    for (;;) {
        const int start = q.ci * chunk_items;
        if (start >= n_items) return n_items;
        const int size = chunk_items < n_items - start ? chunk_items : n_items - start;
        const int wl = q.rd * G + (((q.rd + q.ci) & 1) ? G - 1 - c : c);
        if (wl < size) {
            ++q.rd;
            return start + wl;
        }
        ++q.ci;
        q.rd = 0;
    }
}

struct FwdLaunch {
    CUtensorMap map_q, map_k, map_v;  // 3-D maps (d, N, B*H), box (64, 128, 1), 128B swizzle
    void* o;
    float* lse;
    int B, H, Nq, Nk, d;
    float scale;
    int causal;
    int window;  // > 0: causal sliding window (keys per query)
    const int* lens_q;  // device int32 [B] per-sequence query / key counts, or null (Nq / Nk)
    const int* lens_k;
    int num_sms;
    DevError* err;
    uint64_t timeout_ns;
};

struct BwdLaunch {
    CUtensorMap map_q, map_k, map_v, map_do;  // same geometry as the forward maps
    CUtensorMap map_q2, map_do2;              // d = 128: Q and dO with box (64, 64, 1) (CTA-pair dK/dV pass)
    const void* q;
    const void* k;
    const void* o;
    const void* dO;
    const float* lse;
    void* dq;
    void* dk;
    void* dv;
    float* delta;   // fp32 [B,H,Nq] (the workspace)
    float* dqacc;   // fp32 [B,H,Nq,d] (single-pass backward: zeroed by the preprocess), else null
    int B, H, Nq, Nk, d;
    float scale;
    int causal;
    int window;  // > 0: causal sliding window (keys per query)
    const int* lens_q;  // device int32 [B] per-sequence query / key counts, or null (Nq / Nk)
    const int* lens_k;
    int num_sms;
    DevError* err;
    uint64_t timeout_ns;
};

struct DecodeLaunch {
    const void* q;
    const void* kc;
    const void* vc;
    void* o;
    float* lse;      // may be null
    float* part_o;   // fp32 [B,H,S,d]
    float* part_lse; // fp32 [B,H,S]
    int B, H, Nk, d, splits, chunk;
    float scale;
};

struct PagedDecodeLaunch {
    const void* q;        // bf16 [B, Hq, d]
    const void* kp;       // bf16 [num_pages, Hkv, page, d]
    const void* vp;
    const int* table;     // int32 [B, max_pages]
    const int* lens;      // int32 [B]
    void* o;
    float* lse;           // may be null
    float* part_o;        // fp32 [B, Hq, S, d]
    float* part_lse;      // fp32 [B, Hq, S]
    int B, Hq, Hkv, page, max_pages, num_pages, d, splits;
    float scale;
    DevError* err;
    // tensor-core path only (d = 64 or 128, page a multiple of 8, or the contiguous cache as one page
    // of Nk tokens, a multiple of 128); R = gcd(page, 128) rows per box:
    bool mma;
    CUtensorMap map_q;         // 3-D (d, B*Hq, 1), box (64, 16, 1), 128B swizzle
    CUtensorMap map_k;         // 4-D (d, page, Hkv, num_pages), box (64, R, 1, 1), 128B swizzle; d = 128
                               // with R = 8: map_v's 5-D form (both halves per box)
    CUtensorMap map_v;         // d = 128: 5-D (64, page, 2, Hkv, num_pages), box (64, R, 2, 1, 1);
                               // d = 64: as map_k; 128B swizzle
    int num_sms;
    uint64_t timeout_ns;
};

struct Fp8FwdLaunch {
    CUtensorMap map_q, map_k;  // 3-D uint8 (128, N, B*H), box (128, 128, 1), 128B swizzle
    CUtensorMap map_vt;        // 3-D uint8 (Nk_pad, 128, B*H) over vt, box (128, 128, 1), 128B swizzle
    const void* v;             // e4m3 [B*H, Nk, 128]
    void* vt;                  // workspace: e4m3 [B*H, 128, Nk_pad]
    void* o;                   // bf16 [B*H, Nq, 128]
    float* lse;
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    int B, H, Nq, Nk, Nk_pad;
    float scale;
    int causal;
    int num_sms;
    DevError* err;
    uint64_t timeout_ns;
};

// The dynamic shared-memory limit of kernel K, raised once per device: the
// attribute stays with the function in the context, and setting it costs a
// driver call per launch otherwise.
template <auto K>
cudaError_t set_smem_limit_once(int bytes) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launches kernel k as a programmatic dependent of the kernel before it on
// stream s: its CTAs may start (and run their setup) while that kernel
// finishes.  Every kernel launched this way executes griddepcontrol.wait
// before its first access to global memory, which returns once the kernel
// before it has completed and its writes are visible, and
// griddepcontrol.launch_dependents early, which lets the next one start.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Each returns a cudaError_t of the launch (cudaSuccess when queued).
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t s);
// Whether the plain forward (no window, no per-sequence lengths) takes
// 128-row split-KV tiles for a.B, a.H, a.Nq, a.Nk, a.causal on a.num_sms SMs.
bool fwd_use_split(const FwdLaunch& a);
// Work order of the forward's 256-row tiles (bf16 and FP8): the heads per
// scheduling chunk (*hc) and whether the CTAs take the chunks in per-chunk
// rounds (*per_chunk, next_chunked_item).  hc_l2 heads fill the L2 budget.
// Causal grids take hc_l2-head chunks in per-chunk rounds unless the host's
// replay of both schedules finds the one-chunk, heaviest-first order's
// busiest CTA clearly less loaded; non-causal grids take hc_l2-head chunks in
// rounds over the whole order.
void fwd_work_order(int BH, int Nq, int Nk, int causal, int hc_l2, int num_sms, int* hc, int* per_chunk);
cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t s);   // D = rowsum(dO o O)
cudaError_t launch_bwd_dkdv(const BwdLaunch& a, cudaStream_t s, bool after_pre = false);  // dK, dV; after_pre:
                                                                                        // overlaps the preprocess's end
cudaError_t launch_bwd_dkdv_pair(const BwdLaunch& a, cudaStream_t s);  // dK, dV on CTA pairs (d = 128)
cudaError_t launch_bwd_fused(const BwdLaunch& a, cudaStream_t s);  // dK, dV, dQ in one pass + dQ convert (d = 128)
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t s, bool after_dkdv = false);  // dQ; after_dkdv:
                                                                                     // overlaps the dK/dV grid's end
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t s);
cudaError_t decode_split_blocks_per_sm(int d, int* blocks);  // resident CTAs of the split kernel on one SM
cudaError_t launch_decode_paged(const PagedDecodeLaunch& a, cudaStream_t s);
cudaError_t launch_decode_paged_mma(const PagedDecodeLaunch& a, cudaStream_t s);
cudaError_t launch_fwd_fp8(const Fp8FwdLaunch& a, cudaStream_t s);  // V^T copy, then the forward
// LSE-weighted merge of per-split partials into o (bf16) and lse (fp32, may be null).
cudaError_t launch_decode_combine(const float* part_o, const float* part_lse, void* o, float* lse, int BH,
                                  int splits, int d, cudaStream_t s);

// Rows of the forward's CTA work tile (two 128-row softmax tiles).
constexpr int kFwdRowsPerCta = 256;

}  // namespace fa
