// Split-KV decode: one query token per (b, h) against its KV cache.
//
// The cache stays in HBM and is streamed once (zimaspace.com "Wie reduziert
// Flash Attention den Speicherverkehr ...", section "Weniger IO bedeutet
// nicht, dass der KV-Cache entfällt"); the work is a matrix-vector product,
// bound by HBM bandwidth, so it runs on CUDA cores with 16-byte vector loads.
//
// Kernel 1 (one CTA per (b, h, split), 128 threads): the split's contiguous
// keys are processed in pieces of 128 with the online-softmax update of
// wiki.ai-engineering.at "Flash Attention" ("Lösung: Online Softmax"):
// d/8 lanes share one key row (8 bf16 each), dot products are reduced with
// warp shuffles, the piece maximum with a CTA reduction; partial results are
// the normalised partial output and the partial natural LSE (fp32).
// Kernel 2 (one warp per (b, h)): LSE = M + ln sum_s exp(lse_s - M),
// O = sum_s exp(lse_s - LSE) o_s, rounded to bf16.  An empty split has
// lse_s = -inf and weight 0.
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kDecThreads = 128;
// keys per online-softmax step: 128 at d = 128 (64 KB of K and V in flight per CTA); 256 at
// d = 64, so that a CTA keeps as many bytes in flight and pays its reductions and barriers
// once per 64 KB there too
template <int D>
constexpr int kDecPiece = D == 64 ? 256 : 128;
constexpr int kPagedPiece = 128;  // keys per step of the paged general kernel

template <int D>
__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, float* __restrict__ part_o,
                    float* __restrict__ part_lse, int Nk, int splits, int chunk, float scale_log2) {
    pdl_launch_dependents();
    pdl_wait();  // the cache and q may come from the kernel before; it may still read part_o
    constexpr int PIECE = kDecPiece<D>;
    constexpr int KPT = PIECE / kDecThreads;  // scores per thread in the softmax of a piece
    constexpr int LPK = D / 8;              // lanes per key row
    constexpr int KPW = 32 / LPK;           // keys per warp per load
    constexpr int KPC = KPW * (kDecThreads / 32);  // keys per CTA per load step
    constexpr int STEPS = PIECE / KPC;      // load steps per piece
    __shared__ float s_p[PIECE];
    __shared__ float s_red[kDecThreads / 32];
    __shared__ float s_acc[KPC][D + 4];

    const int split = blockIdx.x % splits;
    const int bh = blockIdx.x / splits;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = lane % LPK;            // which 8 columns of d
    const int group = warp * KPW + lane / LPK;  // key slot within a load step

    const int k0 = split * chunk;
    const int k1 = min(k0 + chunk, Nk);
    float* po = part_o + ((size_t)bh * splits + split) * D;
    if (k0 >= k1) {  // empty split
        if (tid < D / 4) reinterpret_cast<float4*>(po)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid == 0) part_lse[(size_t)bh * splits + split] = -INFINITY;
        return;
    }

    float qf[8];
    {
        const uint4 qv = *reinterpret_cast<const uint4*>(q + (size_t)bh * D + slice * 8);
        const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(q2[i]);
            qf[2 * i] = f.x * scale_log2;  // scores come out in the log2 domain
            qf[2 * i + 1] = f.y * scale_log2;
        }
    }
    const __nv_bfloat16* Kb = kc + (size_t)bh * Nk * D + slice * 8;
    const __nv_bfloat16* Vb = vc + (size_t)bh * Nk * D + slice * 8;

    float m_run = -INFINITY, l_run = 0.f;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;

    for (int p0 = k0; p0 < k1; p0 += PIECE) {
        // ---- scores of this piece (the piece's V rows are loaded with its K rows, so both
        // are in flight together)
        uint4 kr[STEPS], vr[STEPS];
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int key = p0 + s * KPC + group;
            kr[s] = key < k1 ? __ldg(reinterpret_cast<const uint4*>(Kb + (size_t)key * D))
                             : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int key = p0 + s * KPC + group;
            vr[s] = key < k1 ? __ldg(reinterpret_cast<const uint4*>(Vb + (size_t)key * D))
                             : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kr[s]);
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(k2[i]);
                dot = fmaf(qf[2 * i], f.x, dot);
                dot = fmaf(qf[2 * i + 1], f.y, dot);
            }
#pragma unroll
            for (int w = LPK / 2; w >= 1; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
            const int kl = s * KPC + group;
            if (slice == 0) s_p[kl] = (p0 + kl < k1) ? dot : -INFINITY;
        }
        __syncthreads();
        // ---- piece maximum (CTA), new running max; thread tid owns scores tid + 128 i
        float sc[KPT];
#pragma unroll
        for (int i = 0; i < KPT; ++i) sc[i] = s_p[tid + kDecThreads * i];
        float mx = sc[0];
#pragma unroll
        for (int i = 1; i < KPT; ++i) mx = fmaxf(mx, sc[i]);
        for (int w = 16; w >= 1; w >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
        if (lane == 0) s_red[warp] = mx;
        __syncthreads();
        mx = s_red[0];
#pragma unroll
        for (int w = 1; w < kDecThreads / 32; ++w) mx = fmaxf(mx, s_red[w]);
        const float m_new = fmaxf(m_run, mx);  // finite: every piece holds >= 1 key
        const float alpha = ex2(m_run - m_new);  // m_run = -inf on the first piece -> 0
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            sc[i] = ex2(sc[i] - m_new);
            ps += sc[i];
        }
        for (int w = 16; w >= 1; w >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, w);
        __syncthreads();  // s_red, s_p reads done
#pragma unroll
        for (int i = 0; i < KPT; ++i) s_p[tid + kDecThreads * i] = sc[i];
        if (lane == 0) s_red[warp] = ps;
        __syncthreads();
        float psum = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) psum += s_red[w];
        l_run = l_run * alpha + psum;
        m_run = m_new;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] *= alpha;
        // ---- value product of this piece
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const float pj = s_p[s * KPC + group];  // 0 for keys past the split
            const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vr[s]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(v2[i]);
                acc[2 * i] = fmaf(pj, f.x, acc[2 * i]);
                acc[2 * i + 1] = fmaf(pj, f.y, acc[2 * i + 1]);
            }
        }
        __syncthreads();  // s_p / s_red reused by the next piece
    }
    // ---- reduce the KPC key groups, normalise, write the partial
#pragma unroll
    for (int i = 0; i < 8; ++i) s_acc[group][slice * 8 + i] = acc[i];
    __syncthreads();
    const float inv = 1.f / l_run;
    for (int c = tid; c < D; c += kDecThreads) {
        float sum = 0.f;
#pragma unroll
        for (int g = 0; g < KPC; ++g) sum += s_acc[g][c];
        po[c] = sum * inv;
    }
    if (tid == 0) part_lse[(size_t)bh * splits + split] = (m_run + lg2(l_run)) * 0.69314718055994531f;
}

template <int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int BH, int splits) {
    pdl_launch_dependents();
    pdl_wait();  // the partials of the split pass
    constexpr int PER = D / 32;  // output columns per lane
    const int bh = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (bh >= BH) return;
    const float* pl = part_lse + (size_t)bh * splits;
    float M = -INFINITY;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, pl[s]);
    for (int w = 16; w >= 1; w >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, w));
    const float L2E = 1.4426950408889634f;
    float sw = 0.f;
    for (int s = lane; s < splits; s += 32) sw += ex2((pl[s] - M) * L2E);
    for (int w = 16; w >= 1; w >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, w);
    const float LSE = M + lg2(sw) * 0.69314718055994531f;
    float out[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) out[i] = 0.f;
    const float* pob = part_o + (size_t)bh * splits * D + lane * PER;
    for (int s = 0; s < splits; ++s) {
        const float w = ex2((pl[s] - LSE) * L2E);  // exp(-inf) = 0 for an empty split
        if constexpr (PER == 4) {
            const float4 v = *reinterpret_cast<const float4*>(pob + (size_t)s * D);
            out[0] = fmaf(w, v.x, out[0]);
            out[1] = fmaf(w, v.y, out[1]);
            out[2] = fmaf(w, v.z, out[2]);
            out[3] = fmaf(w, v.w, out[3]);
        } else {
            const float2 v = *reinterpret_cast<const float2*>(pob + (size_t)s * D);
            out[0] = fmaf(w, v.x, out[0]);
            out[1] = fmaf(w, v.y, out[1]);
        }
    }
    __nv_bfloat16* ob = o + (size_t)bh * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2)
        *reinterpret_cast<__nv_bfloat162*>(ob + i) = __floats2bfloat162_rn(out[i], out[i + 1]);
    if (lse && lane == 0) lse[bh] = LSE;
}

template <int D>
cudaError_t launch_decode_d(const DecodeLaunch& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    const long long ctas = (long long)BH * a.splits;
    if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    cudaError_t e = launch_dependent(decode_split_kernel<D>, dim3((unsigned)ctas), dim3(kDecThreads), 0, s,
                                     (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kc,
                                     (const __nv_bfloat16*)a.vc, a.part_o, a.part_lse, a.Nk, a.splits, a.chunk,
                                     a.scale * 1.4426950408889634f);
    if (e != cudaSuccess) return e;
    return launch_dependent(decode_combine_kernel<D>, dim3((BH + 3) / 4), dim3(128), 0, s, (const float*)a.part_o,
                            (const float*)a.part_lse, (__nv_bfloat16*)a.o, a.lse, BH, a.splits);
}


// ------------------------------------------------------------------ paged, grouped-query decode
// The general path (page sizes the tensor-core kernel of fa_decode_mma.cu
// does not take: not a multiple of 8).  One CTA per (b,
// kv head, split, group of G <= 4 query heads).  The split's keys are the
// logical tokens [split * chunk, min(len, (split + 1) * chunk)) of the
// sequence, chunk = ceil(len / splits); each 128-key piece's page rows are
// looked up once through the block table (thread = key) into shared memory;
// each K and V row is read once and used for all G query heads of the group
// (they share the kv head).  Same online pieces, partials and combine as the
// contiguous decode.  A page index outside [0, num_pages) or
// a length outside [1, max_pages * page] is recorded as FA_ERR_INVALID_ARG in
// the error word and read as zeros, never dereferenced.
// Resident CTAs per SM the general paged kernel is compiled for.  With four query heads per CTA the
// compiler would otherwise take 168 registers at d = 128 (three CTAs per SM, 0.48 of HBM at
// Hq/Hkv = 4 and 48-token pages); 127 leave four (0.53); five would spill.  The others keep the
// occupancy their register use gives anyway.
template <int D, int G>
constexpr int kPagedMinCtas = G == 4 ? 4 : (D == 128 ? (G == 2 ? 6 : 7) : (G == 2 ? 7 : 10));

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, kPagedMinCtas<D, G>)
decode_paged_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kp,
                          const __nv_bfloat16* __restrict__ vp, const int* __restrict__ table,
                          const int* __restrict__ lens, float* __restrict__ part_o,
                          float* __restrict__ part_lse, int Hq, int Hkv, int page, int max_pages,
                          int num_pages, int splits, int groups, float scale_log2, DevError* err) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int LPK = D / 8, KPW = 32 / LPK, KPC = KPW * (kDecThreads / 32), STEPS = kPagedPiece / KPC;
    __shared__ float s_p[G][kPagedPiece];
    __shared__ float s_red[kDecThreads / 32][G];
    __shared__ float s_acc[KPC][D + 4];
    __shared__ long long s_row[kPagedPiece];  // element offset of each key row of the piece (-1: bad page)
    __shared__ int s_bad;

    int idx = blockIdx.x;
    const int grp = idx % groups; idx /= groups;
    const int split = idx % splits; idx /= splits;
    const int kvh = idx % Hkv;
    const int b = idx / Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = lane % LPK, group = warp * KPW + lane / LPK;
    const int g = Hq / Hkv;
    const int h0 = kvh * g + grp * G;  // first query head of this CTA

    if (tid == 0) s_bad = 0;
    int len = lens[b];
    const int cap = max_pages * page;
    if (len < 1 || len > cap) {
        if (tid == 0 && atomicCAS(&err->code, 0, kErrInvalid) == 0) {
            err->site = kSitePagedTable; err->block = blockIdx.x; err->aux = len;
        }
        len = len < 1 ? 0 : cap;
    }
    const int chunk = (len + splits - 1) / splits;
    const int k0 = split * chunk, k1 = min(k0 + chunk, len);
    if (k0 >= k1) {
        for (int hh = 0; hh < G; ++hh) {
            float* po = part_o + ((size_t)(b * Hq + h0 + hh) * splits + split) * D;
            if (tid < D / 4) reinterpret_cast<float4*>(po)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tid == 0) part_lse[(size_t)(b * Hq + h0 + hh) * splits + split] = -INFINITY;
        }
        return;
    }
    float qf[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const uint4 qv = *reinterpret_cast<const uint4*>(q + (size_t)(b * Hq + h0 + hh) * D + slice * 8);
        const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(q2[i]);
            qf[hh][2 * i] = f.x * scale_log2;
            qf[hh][2 * i + 1] = f.y * scale_log2;
        }
    }
    const int* trow = table + (size_t)b * max_pages;
    float m_run[G], l_run[G], acc[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        m_run[hh] = -INFINITY;
        l_run[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[hh][i] = 0.f;
    }
    bool bad = false;
    for (int p0 = k0; p0 < k1; p0 += kPagedPiece) {
        {   // one block-table lookup per key of the piece (thread = key), shared by the K and V loads
            const int key = p0 + tid;
            long long off = -1;
            if (key < k1) {
                const int pg = trow[key / page];
                if (pg >= 0 && pg < num_pages)
                    off = (((long long)pg * Hkv + kvh) * page + (key % page)) * D;
                else
                    bad = true;
            }
            s_row[tid] = off;
        }
        __syncthreads();
        uint4 kr[STEPS];
#pragma unroll
        for (int s2 = 0; s2 < STEPS; ++s2) {
            const long long off = s_row[s2 * KPC + group];
            kr[s2] = off >= 0 ? __ldg(reinterpret_cast<const uint4*>(kp + off + slice * 8)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int s2 = 0; s2 < STEPS; ++s2) {
            const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kr[s2]);
            float kf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(k2[i]);
                kf[2 * i] = f.x, kf[2 * i + 1] = f.y;
            }
            const int kl = s2 * KPC + group;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) dot = fmaf(qf[hh][i], kf[i], dot);
#pragma unroll
                for (int w = LPK / 2; w >= 1; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
                if (slice == 0) s_p[hh][kl] = (p0 + kl < k1) ? dot : -INFINITY;
            }
        }
        __syncthreads();
        float mx[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float m = s_p[hh][tid];
            for (int w = 16; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, w));
            mx[hh] = m;
        }
        if (lane == 0)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) s_red[warp][hh] = mx[hh];
        __syncthreads();
        float alpha[G], pv[G], ps[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float m = s_red[0][hh];
#pragma unroll
            for (int w = 1; w < kDecThreads / 32; ++w) m = fmaxf(m, s_red[w][hh]);
            const float m_new = fmaxf(m_run[hh], m);
            alpha[hh] = ex2(m_run[hh] - m_new);
            m_run[hh] = m_new;
            pv[hh] = ex2(s_p[hh][tid] - m_new);
            float t = pv[hh];
            for (int w = 16; w >= 1; w >>= 1) t += __shfl_xor_sync(0xffffffffu, t, w);
            ps[hh] = t;
        }
        __syncthreads();
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            s_p[hh][tid] = pv[hh];
            if (lane == 0) s_red[warp][hh] = ps[hh];
        }
        __syncthreads();
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float psum = 0.f;
#pragma unroll
            for (int w = 0; w < kDecThreads / 32; ++w) psum += s_red[w][hh];
            l_run[hh] = l_run[hh] * alpha[hh] + psum;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[hh][i] *= alpha[hh];
        }
        uint4 vr[STEPS];
#pragma unroll
        for (int s2 = 0; s2 < STEPS; ++s2) {
            const long long off = s_row[s2 * KPC + group];
            vr[s2] = off >= 0 ? __ldg(reinterpret_cast<const uint4*>(vp + off + slice * 8)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int s2 = 0; s2 < STEPS; ++s2) {
            const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vr[s2]);
            float vf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(v2[i]);
                vf[2 * i] = f.x, vf[2 * i + 1] = f.y;
            }
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float pj = s_p[hh][s2 * KPC + group];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[hh][i] = fmaf(pj, vf[i], acc[hh][i]);
            }
        }
        __syncthreads();
    }
    if (bad) s_bad = 1;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s_acc[group][slice * 8 + i] = acc[hh][i];
        __syncthreads();
        float* po = part_o + ((size_t)(b * Hq + h0 + hh) * splits + split) * D;
        const float inv = 1.f / l_run[hh];
        for (int c = tid; c < D; c += kDecThreads) {
            float sum = 0.f;
#pragma unroll
            for (int gg = 0; gg < KPC; ++gg) sum += s_acc[gg][c];
            po[c] = sum * inv;
        }
        if (tid == 0)
            part_lse[(size_t)(b * Hq + h0 + hh) * splits + split] = (m_run[hh] + lg2(l_run[hh])) * 0.69314718055994531f;
        __syncthreads();
    }
    if (tid == 0 && s_bad && atomicCAS(&err->code, 0, kErrInvalid) == 0) {
        err->site = kSitePagedTable; err->block = blockIdx.x; err->aux = -1;
    }
}

template <int D, int G>
cudaError_t launch_paged_dg(const PagedDecodeLaunch& a, cudaStream_t s) {
    const int groups = (a.Hq / a.Hkv) / G;
    const long long ctas = (long long)a.B * a.Hkv * a.splits * groups;
    if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    cudaError_t e = launch_dependent(decode_paged_split_kernel<D, G>, dim3((unsigned)ctas), dim3(kDecThreads), 0, s,
                                     (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kp,
                                     (const __nv_bfloat16*)a.vp, a.table, a.lens, a.part_o, a.part_lse, a.Hq,
                                     a.Hkv, a.page, a.max_pages, a.num_pages, a.splits, groups,
                                     a.scale * 1.4426950408889634f, a.err);
    if (e != cudaSuccess) return e;
    const int BH = a.B * a.Hq;
    return launch_dependent(decode_combine_kernel<D>, dim3((BH + 3) / 4), dim3(128), 0, s, (const float*)a.part_o,
                            (const float*)a.part_lse, (__nv_bfloat16*)a.o, a.lse, BH, a.splits);
}

template <int D>
cudaError_t launch_paged_d(const PagedDecodeLaunch& a, cudaStream_t s) {
    const int g = a.Hq / a.Hkv;  // up to 4 query heads per CTA (registers); larger groups use several CTAs
    if (g % 4 == 0) return launch_paged_dg<D, 4>(a, s);
    if (g % 2 == 0) return launch_paged_dg<D, 2>(a, s);
    return launch_paged_dg<D, 1>(a, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_decode_d<128>(a, s) : launch_decode_d<64>(a, s);
}

cudaError_t decode_split_blocks_per_sm(int d, int* blocks) {
    return d == 128 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_split_kernel<128>, kDecThreads, 0)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_split_kernel<64>, kDecThreads, 0);
}

cudaError_t launch_decode_paged(const PagedDecodeLaunch& a, cudaStream_t s) {
    if (a.mma) return launch_decode_paged_mma(a, s);
    return a.d == 128 ? launch_paged_d<128>(a, s) : launch_paged_d<64>(a, s);
}

cudaError_t launch_decode_combine(const float* part_o, const float* part_lse, void* o, float* lse, int BH,
                                  int splits, int d, cudaStream_t s) {
    if (d == 128)
        return launch_dependent(decode_combine_kernel<128>, dim3((BH + 3) / 4), dim3(128), 0, s, part_o, part_lse,
                                (__nv_bfloat16*)o, lse, BH, splits);
    return launch_dependent(decode_combine_kernel<64>, dim3((BH + 3) / 4), dim3(128), 0, s, part_o, part_lse,
                            (__nv_bfloat16*)o, lse, BH, splits);
}

}  // namespace fa
