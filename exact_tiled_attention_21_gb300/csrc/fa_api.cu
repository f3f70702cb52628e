// The C ABI declared in include/fa.h: argument validation, TMA tensor-map
// encoding, the per-device error word, and the launches.  No allocation, no
// fallback: every call either launches the GPU kernels or returns an error.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ DevError g_dev_error;  // one per device (per context)

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::mutex g_mu;
DevError* g_err_addr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device state, looked up with the current device active.
int device_state(DevError** err, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_addr[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_dev_error) != cudaSuccess || !a) return FA_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            return FA_ERR_CUDA;
        g_err_addr[dev] = static_cast<DevError*>(a);
        g_num_sms[dev] = sms;
    }
    if (err) *err = g_err_addr[dev];
    if (num_sms) *num_sms = g_num_sms[dev];
    return FA_OK;
}

int encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return FA_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    *fn = g_encode;
    return FA_OK;
}

// 3-D map over a contiguous (BH, N, d) bf16 tensor: dims (d, N, BH), box
// (64, 128, 1), 128-byte swizzle (matches the MMA shared-memory descriptors).
int make_map(CUtensorMap* m, const void* base, int BH, int N, int d, unsigned box_rows = 128) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int st = encoder(&enc);
    if (st != FA_OK) return st;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Tiled map of any rank (bf16, 128-byte swizzle, zero fill out of range).
// strides: bytes of dims 1..rank-1.
int make_map_nd(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int st = encoder(&enc);
    if (st != FA_OK) return st;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, dtype, rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// Page sizes the tensor-core paged decode takes: whole 8-row swizzle atoms per page.  It loads
// a page in boxes of gcd(page, 128) rows (at least 8), which tile both the page and a 128-key
// stage.
bool paged_mma_ok(int d, int page) { return (d == 64 || d == 128) && page % 8 == 0; }

// Rows of one TMA box of a page: gcd(page, 128) for a multiple of 8.
int page_box_rows(int page) { return std::min(page & -page, 128); }

// Shared shape checks.  Sizes must keep every element index below 2^31 per
// tensor row block and the total within 64-bit byte offsets.
int check_shape(int B, int H, int Nq, int Nk, int d) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const long long BH = (long long)B * H;
    if (BH > (1ll << 24)) return FA_ERR_UNSUPPORTED;  // work-tile indices stay in int
    if ((long long)Nq * BH > (1ll << 36) || (long long)Nk * BH > (1ll << 36)) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// The backward keeps dQ in TMEM (Q-tile-parallel pass), so its only scratch
// is D = rowsum(dO o O): one fp32 per query row.
size_t bwd_ws_bytes(int B, int H, int Nq, int d) {
    (void)d;
    const size_t rows = (size_t)B * H * Nq;
    return (rows * 4 + 255) & ~(size_t)255;
}

int decode_auto_splits(int Nk) {
    // chunks of at least 256 keys, at most 16 chunks
    int s = (Nk + 255) / 256;
    return s < 1 ? 1 : (s > 16 ? 16 : s);
}

int g_dec_blocks[kMaxDevices][2] = {};  // resident split-kernel CTAs per SM, by device and d (64, 128)

// Automatic split count of the contiguous decode on CUDA cores.  One CTA per (b, h, split) keeps a
// fixed number of loads in flight, so a launch costs about waves * (per-CTA time): waves =
// ceil(B*H*splits / resident CTAs), per-CTA time = the split's key pieces plus a fixed cost of
// about one piece (q load, reductions, the partial write), in keys.  Among 1 .. decode_auto_splits(Nk)
// splits it takes the cheapest, the fewest on a tie (fewer partials to merge).  A split count
// that spills a few CTAs into a second wave costs a whole wave: at B=8, H=32, Nk=4000, d=128 (7
// CTAs per SM, 1064 resident) 4 splits read 0.83 of HBM and 6 splits 0.68.
int decode_wave_splits(int B, int H, int Nk, int d, int* splits) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    int num_sms = 0;
    int st = device_state(nullptr, &num_sms);
    if (st != FA_OK) return st;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int& c = g_dec_blocks[dev][d == 128 ? 1 : 0];
        if (!c) {
            int b = 0;
            if (decode_split_blocks_per_sm(d, &b) != cudaSuccess || b < 1) return FA_ERR_CUDA;
            c = b;
        }
        per_sm = c;
    }
    const long long resident = (long long)num_sms * per_sm, bh = (long long)B * H;
    const long long piece = d == 64 ? 256 : 128;  // keys per online-softmax step of the kernel
    const int cap = decode_auto_splits(Nk);
    int best = cap;
    long long best_cost = LLONG_MAX;
    for (int sp = 1; sp <= cap; ++sp) {
        const long long chunk = (Nk + sp - 1) / sp;
        const long long waves = (bh * sp + resident - 1) / resident;
        const long long cost = waves * ((chunk + piece - 1) / piece * piece + 128);
        if (cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    *splits = best;
    return FA_OK;
}

// Paged decode, automatic splits.  The lengths live on the device, so the host
// plans for the longest possible sequence (max_pages * page).  The tensor-core
// kernel is persistent: items = B * Hkv * (head groups) * splits are dealt to
// the SMs round-robin.  Its cost model is waves * (1/splits + 0.02): a split
// is a share of the sequence plus a fixed per-item overhead.  It picks the
// best of 1..16 splits with at least 128 keys each.  The general kernel uses
// the contiguous decode's rule.
int paged_auto_splits(int B, int Hq, int Hkv, int max_len, int num_sms, bool mma) {
    if (!mma) return decode_auto_splits(max_len);
    const int g = Hq / Hkv;
    const int nh = g <= 4 ? 4 : (g <= 8 ? 8 : 16);
    const long long base = (long long)B * Hkv * ((g + nh - 1) / nh);
    int best = 1;
    double best_cost = 1e30;
    for (int sp = 1; sp <= 16 && (sp == 1 || (long long)sp * 128 <= max_len); ++sp) {
        const long long waves = (base * sp + num_sms - 1) / num_sms;
        const double cost = (double)waves * (1.0 / sp + 0.02);
        if (cost < best_cost - 1e-12) {
            best_cost = cost;
            best = sp;
        }
    }
    return best;
}

size_t decode_ws_bytes(int B, int H, int d, int splits) {
    const size_t parts = (size_t)B * H * splits;
    return parts * d * 4 + ((parts * 4 + 255) & ~(size_t)255);
}

// Watchdog self-test: one thread waits on an mbarrier that nothing ever
// arrives on.  The bounded wait gives up after `timeout_ns`, records
// FA_ERR_TIMEOUT at kSiteProbe in the error word and the kernel returns.
__global__ void selftest_wait_kernel(DevError* err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const WaitCtl ctl{err, timeout_ns, &abort_flag};
    mbar_wait(b, 0, ctl, kSiteProbe);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

uint64_t fa_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 1000000ull) ns = 1000000ull;
    return g_timeout_ns.exchange(ns);
}

const char* fa_status_string(int st) {
    switch (st) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128)";
        case FA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case FA_ERR_WORKSPACE: return "workspace missing or too small";
        case FA_ERR_CUDA: return "CUDA call failed";
        case FA_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"

namespace {
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
             int d, float scale, int causal, int window, const int* lens_q, const int* lens_k, void* stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, Nq, Nk, d);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_ALIGNMENT;
    if ((lens_q && !aligned4(lens_q)) || (lens_k && !aligned4(lens_k))) return FA_ERR_ALIGNMENT;
    FwdLaunch a;
    st = device_state(&a.err, &a.num_sms);
    if (st != FA_OK) return st;
    const int BH = B * H;
    if (make_map(&a.map_q, q, BH, Nq, d) || make_map(&a.map_k, k, BH, Nk, d) ||
        make_map(&a.map_v, v, BH, Nk, d))
        return FA_ERR_CUDA;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.window = window;
    a.lens_q = lens_q;
    a.lens_k = lens_k;
    a.timeout_ns = g_timeout_ns.load();
    return launch_fwd(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
           int Nk, int d, float scale, int causal, void* stream) {
    return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 0, nullptr, nullptr, stream);
}

int fa_work_schedule(int n_items, int chunk_items, int grid, int per_chunk, int* owner) {
    if (n_items < 0 || chunk_items < 1 || grid < 1 || (n_items > 0 && !owner)) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < n_items; ++i) owner[i] = -1;
    for (int c = 0; c < grid; ++c) {
        ItemSeq q;
        for (int w = next_chunked_item(q, n_items, chunk_items, grid, c, per_chunk != 0); w < n_items;
             w = next_chunked_item(q, n_items, chunk_items, grid, c, per_chunk != 0)) {
            if (w < 0 || owner[w] != -1) return FA_ERR_INVALID_ARG;
            owner[w] = c;
        }
    }
    return FA_OK;
}

int fa_fwd_tile_rows(int B, int H, int Nq, int Nk, int d, int causal) {
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, Nq, Nk, d);
    if (st != FA_OK) return st;
    FwdLaunch a;
    st = device_state(&a.err, &a.num_sms);
    if (st != FA_OK) return st;
    a.B = B;
    a.H = H;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.causal = causal;
    return fwd_use_split(a) ? 128 : kFwdRowsPerCta;
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* seqlens_q,
                  const int* seqlens_k, int B, int H, int Nq, int Nk, int d, float scale, int causal, void* stream) {
    if (!seqlens_q || !seqlens_k) return FA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 0, seqlens_q, seqlens_k, stream);
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                  int Nk, int d, float scale, int window, void* stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, 1, window, nullptr, nullptr, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
    if (check_shape(B, H, Nq, Nk, d) != FA_OK) return 0;
    return bwd_ws_bytes(B, H, Nq, d);
}

size_t fa_bwd_fused_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
    if (check_shape(B, H, Nq, Nk, d) != FA_OK || d != 128) return 0;
    return bwd_ws_bytes(B, H, Nq, d) + (((size_t)B * H * Nq * d * 4 + 255) & ~(size_t)255);
}

}  // extern "C"

namespace {

// Shared checks of the backward steps.  Pointers that a step does not use are
// passed as `used = false` and not checked.
int bwd_prepare(BwdLaunch* a, const void* q, const void* k, const void* v, const void* o, const float* lse,
                const float* delta, const void* dO, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk,
                int d, float scale, int causal, bool need_maps) {
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, Nq, Nk, d);
    if (st != FA_OK) return st;
    const void* ptrs[] = {q, k, v, o, lse, delta, dO, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return FA_ERR_ALIGNMENT;
    st = device_state(&a->err, &a->num_sms);
    if (st != FA_OK) return st;
    const int BH = B * H;
    if (need_maps && (make_map(&a->map_q, q, BH, Nq, d) || make_map(&a->map_k, k, BH, Nk, d) ||
                      make_map(&a->map_v, v, BH, Nk, d) || make_map(&a->map_do, dO, BH, Nq, d)))
        return FA_ERR_CUDA;
    if (need_maps && d == 128 && (make_map(&a->map_q2, q, BH, Nq, d, 64) || make_map(&a->map_do2, dO, BH, Nq, d, 64)))
        return FA_ERR_CUDA;
    a->q = q;
    a->k = k;
    a->o = o;
    a->dO = dO;
    a->lse = lse;
    a->dq = dq;
    a->dk = dk;
    a->dv = dv;
    a->delta = const_cast<float*>(delta);
    a->dqacc = nullptr;
    a->B = B;
    a->H = H;
    a->Nq = Nq;
    a->Nk = Nk;
    a->d = d;
    a->scale = scale;
    a->causal = causal;
    a->window = 0;
    a->lens_q = nullptr;
    a->lens_k = nullptr;
    a->timeout_ns = g_timeout_ns.load();
    return FA_OK;
}

int launched(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
             int window, const int* lens_q, const int* lens_k, void* workspace, size_t workspace_bytes,
             void* stream, bool fused = false) {
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if ((lens_q && !aligned4(lens_q)) || (lens_k && !aligned4(lens_k))) return FA_ERR_ALIGNMENT;
    int st = check_shape(B, H, Nq, Nk, d);
    if (st != FA_OK) return st;
    if (fused && d != 128) return FA_ERR_UNSUPPORTED;
    const size_t ws_need = fused ? fa_bwd_fused_workspace_bytes(B, H, Nq, Nk, d) : bwd_ws_bytes(B, H, Nq, d);
    if (!workspace || workspace_bytes < ws_need) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
    BwdLaunch a;
    st = bwd_prepare(&a, q, k, v, o, lse, static_cast<float*>(workspace), dO, dq, dk, dv, B, H, Nq, Nk, d,
                     scale, causal, true);
    if (st != FA_OK) return st;
    a.window = window;
    a.lens_q = lens_q;
    a.lens_k = lens_k;
    cudaStream_t s = (cudaStream_t)stream;
    if (fused) {  // the fp32 dQ accumulator follows D in the workspace
        a.dqacc = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_ws_bytes(B, H, Nq, d));
        if ((st = launched(launch_bwd_pre(a, s))) != FA_OK) return st;
        return launched(launch_bwd_fused(a, s));
    }
    if ((st = launched(launch_bwd_pre(a, s))) != FA_OK) return st;
    if ((st = launched(launch_bwd_dkdv(a, s, true))) != FA_OK) return st;
    return launched(launch_bwd_dq(a, s, true));
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
           void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
           void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, 0, nullptr, nullptr,
                    workspace, workspace_bytes, stream);
}

int fa_bwd_fused(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, 0, nullptr, nullptr,
                    workspace, workspace_bytes, stream, true);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, const int* seqlens_q, const int* seqlens_k, int B, int H, int Nq,
                  int Nk, int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!seqlens_q || !seqlens_k) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, 0, seqlens_q, seqlens_k,
                    workspace, workspace_bytes, stream);
}

int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int window,
                  void* workspace, size_t workspace_bytes, void* stream) {
    if (window < 1) return FA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, 1, window, nullptr, nullptr,
                    workspace, workspace_bytes, stream);
}

int fa_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int H, int Nq, int d, void* stream) {
    if (!o || !dO || !delta) return FA_ERR_INVALID_ARG;
    BwdLaunch a;
    int st = bwd_prepare(&a, nullptr, nullptr, nullptr, o, nullptr, delta, dO, nullptr, nullptr, nullptr, B, H,
                         Nq, 1, d, 1.f, 0, false);
    if (st != FA_OK) return st;
    return launched(launch_bwd_pre(a, (cudaStream_t)stream));
}

int fa_bwd_dkdv(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                const void* dO, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                void* stream) {
    if (!q || !k || !v || !lse || !delta || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
    BwdLaunch a;
    int st = bwd_prepare(&a, q, k, v, nullptr, lse, delta, dO, nullptr, dk, dv, B, H, Nq, Nk, d, scale, causal,
                         true);
    if (st != FA_OK) return st;
    return launched(launch_bwd_dkdv(a, (cudaStream_t)stream));
}

int fa_bwd_dkdv_pair(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                     const void* dO, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale,
                     int causal, void* stream) {
    if (!q || !k || !v || !lse || !delta || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (d == 64) return FA_ERR_UNSUPPORTED;  // other d: the shape check below
    BwdLaunch a;
    int st = bwd_prepare(&a, q, k, v, nullptr, lse, delta, dO, nullptr, dk, dv, B, H, Nq, Nk, d, scale, causal,
                         true);
    if (st != FA_OK) return st;
    return launched(launch_bwd_dkdv_pair(a, (cudaStream_t)stream));
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const float* lse, const float* delta, const void* dO,
              void* dq, int B, int H, int Nq, int Nk, int d, float scale, int causal, void* stream) {
    if (!q || !k || !v || !lse || !delta || !dO || !dq) return FA_ERR_INVALID_ARG;
    BwdLaunch a;
    int st = bwd_prepare(&a, q, k, v, nullptr, lse, delta, dO, dq, nullptr, nullptr, B, H, Nq, Nk, d, scale,
                         causal, true);
    if (st != FA_OK) return st;
    return launched(launch_bwd_dq(a, (cudaStream_t)stream));
}

size_t fa_decode_workspace_bytes(int B, int H, int Nk, int d, int num_splits) {
    if (check_shape(B, H, 1, Nk, d) != FA_OK || num_splits > 256) return 0;
    const int s = num_splits <= 0 ? decode_auto_splits(Nk) : num_splits;
    return decode_ws_bytes(B, H, d, s);
}

}  // extern "C"

namespace {

// Tensor maps of the tensor-core paged decode (d = 128): q, and K/V as pages.
int paged_mma_maps(PagedDecodeLaunch& a) {
    const int d = a.d, page_size = a.page;
    const cuuint64_t qd[3] = {(cuuint64_t)d, (cuuint64_t)a.B * a.Hq, 1};
    const cuuint64_t qs[2] = {(cuuint64_t)d * 2, (cuuint64_t)a.B * a.Hq * d * 2};
    const cuuint32_t qb[3] = {64, 16, 1};
    const cuuint64_t kd[4] = {(cuuint64_t)d, (cuuint64_t)page_size, (cuuint64_t)a.Hkv, (cuuint64_t)a.num_pages};
    const cuuint64_t ks[3] = {(cuuint64_t)d * 2, (cuuint64_t)page_size * d * 2,
                              (cuuint64_t)a.Hkv * page_size * d * 2};
    const cuuint32_t kb[4] = {64, (cuuint32_t)page_box_rows(page_size), 1, 1};
    // V: the feature dimension as (64, half) so one box holds a page's rows of both halves
    const cuuint64_t vd[5] = {64, (cuuint64_t)page_size, 2, (cuuint64_t)a.Hkv, (cuuint64_t)a.num_pages};
    const cuuint64_t vs[4] = {(cuuint64_t)d * 2, 128, (cuuint64_t)page_size * d * 2,
                              (cuuint64_t)a.Hkv * page_size * d * 2};
    const cuuint32_t vb[5] = {64, (cuuint32_t)page_box_rows(page_size), 2, 1, 1};
    // d = 64: a row is one 128-byte swizzle row, so V takes the same 4-D form as K.  d = 128 with
    // 8-row boxes: K takes V's 5-D form too (one copy per box for both feature halves; the kernel
    // addresses the halves 1 KB apart and the 8-row groups 2 KB apart)
    const bool k5 = d == 128 && page_box_rows(page_size) == 8;
    if (make_map_nd(&a.map_q, a.q, 3, qd, qs, qb) ||
        (k5 ? make_map_nd(&a.map_k, a.kp, 5, vd, vs, vb) : make_map_nd(&a.map_k, a.kp, 4, kd, ks, kb)) ||
        (d == 128 ? make_map_nd(&a.map_v, a.vp, 5, vd, vs, vb) : make_map_nd(&a.map_v, a.vp, 4, kd, ks, kb)))
        return FA_ERR_CUDA;
    return FA_OK;
}

// Contiguous decode (fa_decode, fa_decode_noalloc) with d = 128 and Nk a multiple of 128 runs on the
// tensor-core paged kernel: the cache [B, H, Nk, d] is the paged layout with one page of Nk tokens per
// sequence (page b of sequence b, implicit in the kernel), one kv head per query head.  Its TMA stages
// read the cache at ~6.8 TB/s against ~6.3 TB/s for the 16-byte-load kernel.  Other shapes are faster
// on the 16-byte-load kernel (measured at B=32, H=32, 16 splits): with one query head per kv head
// every work item is a split of two 128-key stages, and the kernel's fixed cost per item and per
// stage, which d = 128 hides behind 64 KB of cache per stage, shows at d = 64 (4.0 against 5.8 TB/s
// at Nk = 4096) and on a ragged last stage (6.0 against 6.2 TB/s at Nk = 4000).  Returns false when
// the shape takes the 16-byte-load kernel.
bool contiguous_on_mma(int Nk, int d) { return d == 128 && Nk % 128 == 0 && paged_mma_ok(d, Nk); }

int launch_contiguous_on_mma(const void* q, const void* kcache, const void* vcache, void* o, float* lse, int B,
                             int H, int Nk, int d, float scale, int splits, float* part_o, void* stream) {
    PagedDecodeLaunch a;
    int st = device_state(&a.err, &a.num_sms);
    if (st != FA_OK) return st;
    a.mma = true;
    a.q = q;
    a.kp = kcache;
    a.vp = vcache;
    a.table = nullptr;
    a.lens = nullptr;
    a.o = o;
    a.lse = lse;
    a.part_o = part_o;
    a.part_lse = part_o + (size_t)B * H * splits * d;  // the layout of the fa_decode workspace
    a.B = B;
    a.Hq = H;
    a.Hkv = H;
    a.page = Nk;
    a.max_pages = 1;
    a.num_pages = B;
    a.d = d;
    a.splits = splits;
    a.scale = scale;
    a.timeout_ns = g_timeout_ns.load();
    st = paged_mma_maps(a);
    if (st != FA_OK) return st;
    return launch_decode_paged(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_decode(const void* q, const void* kcache, const void* vcache, void* o, float* lse, int B, int H,
              int Nk, int d, float scale, int num_splits, void* workspace, size_t workspace_bytes,
              void* stream) {
    if (!q || !kcache || !vcache || !o) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale) || num_splits > 256) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, 1, Nk, d);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return FA_ERR_ALIGNMENT;
    // automatic: the tensor-core path reads best with the most splits its length allows; the
    // CUDA-core kernel takes the wave rule above.  Both stay within decode_auto_splits(Nk), the
    // count fa_decode_workspace_bytes sizes for.
    int splits = num_splits <= 0 ? decode_auto_splits(Nk) : num_splits;
    if (num_splits <= 0 && !contiguous_on_mma(Nk, d)) {
        st = decode_wave_splits(B, H, Nk, d, &splits);
        if (st != FA_OK) return st;
    }
    if (!workspace || workspace_bytes < decode_ws_bytes(B, H, d, splits)) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
    if (contiguous_on_mma(Nk, d))
        return launch_contiguous_on_mma(q, kcache, vcache, o, lse, B, H, Nk, d, scale, splits,
                                        static_cast<float*>(workspace), stream);
    st = device_state(nullptr, nullptr);
    if (st != FA_OK) return st;
    DecodeLaunch a;
    a.q = q;
    a.kc = kcache;
    a.vc = vcache;
    a.o = o;
    a.lse = lse;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = a.part_o + (size_t)B * H * splits * d;
    a.B = B;
    a.H = H;
    a.Nk = Nk;
    a.d = d;
    a.splits = splits;
    a.chunk = (Nk + splits - 1) / splits;
    a.scale = scale;
    return launch_decode(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_decode_paged_workspace_bytes(int B, int Hq, int d, int num_splits) {
    if (B < 1 || Hq < 1 || (d != 64 && d != 128) || num_splits > 256) return 0;
    return decode_ws_bytes(B, Hq, d, num_splits <= 0 ? 16 : num_splits);  // automatic: at most 16
}

int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                    const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int page_size,
                    int max_pages, int num_pages, int d, float scale, int num_splits, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale) || num_splits > 256) return FA_ERR_INVALID_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || page_size < 1 || max_pages < 1 || num_pages < 1) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size > 0x7FFFFFFFll || (long long)B * Hq > (1ll << 24)) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || (lse && !aligned16(lse)) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return FA_ERR_ALIGNMENT;
    PagedDecodeLaunch a;
    int st = device_state(&a.err, &a.num_sms);
    if (st != FA_OK) return st;
    a.mma = paged_mma_ok(d, page_size);
    if (num_splits <= 0)
        num_splits = paged_auto_splits(B, Hq, Hkv, max_pages * page_size, a.num_sms, a.mma);
    if (!workspace || workspace_bytes < decode_ws_bytes(B, Hq, d, num_splits)) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
    a.q = q;
    a.kp = k_pages;
    a.vp = v_pages;
    a.table = block_table;
    a.lens = seq_lens;
    a.o = o;
    a.lse = lse;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = a.part_o + (size_t)B * Hq * num_splits * d;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.page = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.d = d;
    a.splits = num_splits;
    a.scale = scale;
    if (a.mma) {
        a.timeout_ns = g_timeout_ns.load();
        st = paged_mma_maps(a);
        if (st != FA_OK) return st;
    }
    return launch_decode_paged(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Nk, int d) {
    if (B < 1 || H < 1 || Nk < 1 || d != 128 || (long long)B * H > (1ll << 24)) return 0;
    const size_t nk_pad = ((size_t)Nk + 15) & ~(size_t)15;
    return (((size_t)B * H * 128 * nk_pad) + 255) & ~(size_t)255;
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int Nq, int Nk, int d, float scale,
               int causal, void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !o || !lse) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, Nq, Nk, d);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale))
        return FA_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < fa_fwd_fp8_workspace_bytes(B, H, Nk, d)) return FA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
    Fp8FwdLaunch a;
    st = device_state(&a.err, &a.num_sms);
    if (st != FA_OK) return st;
    const cuuint64_t BH = (cuuint64_t)B * H;
    const int nk_pad = (Nk + 15) & ~15;
    const cuuint32_t box[3] = {128, 128, 1};
    const cuuint64_t qd[3] = {128, (cuuint64_t)Nq, BH}, qs[2] = {128, (cuuint64_t)Nq * 128};
    const cuuint64_t kd[3] = {128, (cuuint64_t)Nk, BH}, ks[2] = {128, (cuuint64_t)Nk * 128};
    const cuuint64_t vd[3] = {(cuuint64_t)nk_pad, 128, BH}, vs[2] = {(cuuint64_t)nk_pad, (cuuint64_t)nk_pad * 128};
    if (make_map_nd(&a.map_q, q, 3, qd, qs, box, CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        make_map_nd(&a.map_k, k, 3, kd, ks, box, CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        make_map_nd(&a.map_vt, workspace, 3, vd, vs, box, CU_TENSOR_MAP_DATA_TYPE_UINT8))
        return FA_ERR_CUDA;
    a.v = v;
    a.vt = workspace;
    a.o = o;
    a.lse = lse;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.B = B;
    a.H = H;
    a.Nq = Nq;
    a.Nk = Nk;
    a.Nk_pad = nk_pad;
    a.scale = scale;
    a.causal = causal;
    a.timeout_ns = g_timeout_ns.load();
    return launch_fwd_fp8(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return FA_ERR_INVALID_ARG;
    DevError* err = nullptr;
    int st = device_state(&err, nullptr);
    if (st != FA_OK) return st;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_get_last_device_error(void* stream, int* detail) {
    if (detail)
        for (int i = 0; i < 4; ++i) detail[i] = 0;
    DevError* err = nullptr;
    if (device_state(&err, nullptr) != FA_OK) return FA_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FA_ERR_CUDA;
    DevError h;
    if (cudaMemcpy(&h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (h.code != 0) {
        DevError z = {0, 0, 0, 0};
        if (cudaMemcpy(err, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (detail) {
        detail[0] = h.code;
        detail[1] = h.site;
        detail[2] = h.block;
        detail[3] = h.aux;
    }
    return h.code;  // FA_OK, or the first code a kernel recorded
}

}  // extern "C"

// ---------------------------------------------------------------- decode without a workspace
// fa_decode_noalloc: the split partials live in one fixed array compiled into
// the library, for callers that may not allocate device memory (see fa.h).
// In host code the name of the array is only a stand-in; its device address
// comes from cudaGetSymbolAddress, looked up once per device with that device
// current, and is what the kernels receive.
static __device__ __align__(256) unsigned char g_fa_decode_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[fa::kMaxDevices] = {};
}  // namespace

extern "C" int fa_decode_noalloc(const void* q, const void* kcache, const void* vcache, void* o, float* lse,
                                 int B, int H, int Nk, int d, float scale, int num_splits, void* stream) {
    if (!q || !kcache || !vcache || !o) return FA_ERR_INVALID_ARG;
    if (!scale_ok(scale) || num_splits > 256) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, 1, Nk, d);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        (lse && !aligned16(lse)))
        return FA_ERR_ALIGNMENT;
    int splits = num_splits <= 0 ? decode_auto_splits(Nk) : num_splits;  // the rule of fa_decode
    if (num_splits <= 0 && !contiguous_on_mma(Nk, d)) {
        st = decode_wave_splits(B, H, Nk, d, &splits);
        if (st != FA_OK) return st;
    }
    if (decode_ws_bytes(B, H, d, splits) > FA_DECODE_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_fa_decode_scratch) != cudaSuccess || !addr) return FA_ERR_CUDA;
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    if (contiguous_on_mma(Nk, d))
        return launch_contiguous_on_mma(q, kcache, vcache, o, lse, B, H, Nk, d, scale, splits,
                                        static_cast<float*>(scratch), stream);
    DecodeLaunch a;
    a.q = q;
    a.kc = kcache;
    a.vc = vcache;
    a.o = o;
    a.lse = lse;
    a.part_o = static_cast<float*>(scratch);
    a.part_lse = a.part_o + (size_t)B * H * splits * d;  // same layout as the fa_decode workspace
    a.B = B;
    a.H = H;
    a.Nk = Nk;
    a.d = d;
    a.splits = splits;
    a.chunk = (Nk + splits - 1) / splits;
    a.scale = scale;
    return launch_decode(a, (cudaStream_t)stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
