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
constexpr int kDecPiece = 128;  // keys per online-softmax step

template <int D>
__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, float* __restrict__ part_o,
                    float* __restrict__ part_lse, int Nk, int splits, int chunk, float scale_log2) {
    constexpr int LPK = D / 8;              // lanes per key row
    constexpr int KPW = 32 / LPK;           // keys per warp per load
    constexpr int KPC = KPW * (kDecThreads / 32);  // keys per CTA per load step
    constexpr int STEPS = kDecPiece / KPC;  // load steps per piece
    __shared__ float s_p[kDecPiece];
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

    for (int p0 = k0; p0 < k1; p0 += kDecPiece) {
        // ---- scores of this piece
        uint4 kr[STEPS];
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int key = p0 + s * KPC + group;
            kr[s] = key < k1 ? __ldg(reinterpret_cast<const uint4*>(Kb + (size_t)key * D))
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
        // ---- piece maximum (CTA), new running max
        float mx = s_p[tid];  // kDecThreads == kDecPiece
        for (int w = 16; w >= 1; w >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
        if (lane == 0) s_red[warp] = mx;
        __syncthreads();
        mx = s_red[0];
#pragma unroll
        for (int w = 1; w < kDecThreads / 32; ++w) mx = fmaxf(mx, s_red[w]);
        const float m_new = fmaxf(m_run, mx);  // finite: every piece holds >= 1 key
        const float alpha = ex2(m_run - m_new);  // m_run = -inf on the first piece -> 0
        const float pv = ex2(s_p[tid] - m_new);
        float ps = pv;
        for (int w = 16; w >= 1; w >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, w);
        __syncthreads();  // s_red, s_p reads done
        s_p[tid] = pv;
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
        uint4 vr[STEPS];
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int key = p0 + s * KPC + group;
            vr[s] = key < k1 ? __ldg(reinterpret_cast<const uint4*>(Vb + (size_t)key * D))
                             : make_uint4(0, 0, 0, 0);
        }
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
    decode_split_kernel<D><<<(unsigned)ctas, kDecThreads, 0, s>>>(
        (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kc, (const __nv_bfloat16*)a.vc, a.part_o,
        a.part_lse, a.Nk, a.splits, a.chunk, a.scale * 1.4426950408889634f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D><<<(BH + 3) / 4, 128, 0, s>>>(a.part_o, a.part_lse, (__nv_bfloat16*)a.o,
                                                          a.lse, BH, a.splits);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t s) {
    return a.d == 128 ? launch_decode_d<128>(a, s) : launch_decode_d<64>(a, s);
}

}  // namespace fa
