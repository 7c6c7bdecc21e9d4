// Block Attention Residual (AttnRes) aggregation: the input of a later layer
// as attention over depth of M block summaries, token by token:
//
//     k_n(t) = s_n(t) / sqrt(mean_c s_n(t, c)^2 + eps)
//     a_n(t) = softmax over n of (w . k_n(t))
//     x(t)   = sum_n a_n(t) s_n(t)
//
// "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section "Architecture")
// names a shared, timestep-independent Attention Residual aggregation in
// blocks of eight layers; the arXiv abstract of 2607.21553 says completed
// block summaries are routed into later linear layers.  The formula above is
// a reading (the pages print none): one learned query w shared by all tokens,
// RMS-normalised summaries as keys, the raw summaries as values.
//
// HBM-bound: every summary row is read once from HBM and x written once.  One
// warp per token: the first pass reads the M rows (512 contiguous bytes per
// warp load) and forms w . s_n and s_n . s_n; after the warp reductions and
// the softmax, the second pass reads the same rows again, from L2 (the warps
// in flight hold a few MB), and writes x.
#include "launch.h"

namespace sla {
namespace {

constexpr int kArWarps = 8;                 // tokens per 256-thread block

struct AttnResParams {
    const __nv_bfloat16* src[kAttnResMaxSources];
    int M;
    int C;                                  // a multiple of 256
    long long T;
    float eps;
    const float* w;
    __nv_bfloat16* out;
};

__device__ __forceinline__ void unpack8(uint4 u, float (&x)[8]) {
    const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = bf2_to_f2(v[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// 16-byte global load kept in L2 for the second pass, not allocated in L1.
__device__ __forceinline__ uint4 ld_keep(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(reinterpret_cast<uint64_t>(p)));
    return v;
}

// The second read of a row: its last use, so L2 may evict it first.
__device__ __forceinline__ uint4 ld_last(const void* p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(reinterpret_cast<uint64_t>(p)), "l"(policy));
    return v;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__global__ void __launch_bounds__(kArWarps * 32)
attnres_kernel(AttnResParams p) {
    extern __shared__ float ws[];           // w, C floats
    for (int i = threadIdx.x; i < p.C; i += blockDim.x) ws[i] = __ldg(p.w + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const long long t = (long long)blockIdx.x * kArWarps + (threadIdx.x >> 5);
    if (t >= p.T) return;
    const int chunks = p.C >> 8;            // 256 columns: 8 per lane
    const size_t row = (size_t)t * p.C + (size_t)lane * 8;

    float dot[kAttnResMaxSources], ss[kAttnResMaxSources];
#pragma unroll
    for (int n = 0; n < kAttnResMaxSources; ++n) {
        dot[n] = 0.f;
        ss[n] = 0.f;
        if (n < p.M) {
            const __nv_bfloat16* s = p.src[n] + row;
#pragma unroll 4
            for (int ch = 0; ch < chunks; ++ch) {
                float x[8];
                unpack8(ld_keep(s + ch * 256), x);
                const float4 w0 = *reinterpret_cast<const float4*>(ws + ch * 256 + lane * 8);
                const float4 w1 = *reinterpret_cast<const float4*>(ws + ch * 256 + lane * 8 + 4);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    dot[n] = fmaf(x[i], wv[i], dot[n]);
                    ss[n] = fmaf(x[i], x[i], ss[n]);
                }
            }
        }
    }
#pragma unroll
    for (int n = 0; n < kAttnResMaxSources; ++n) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            dot[n] += __shfl_xor_sync(0xffffffffu, dot[n], off);
            ss[n] += __shfl_xor_sync(0xffffffffu, ss[n], off);
        }
    }
    // a_n = softmax_n(dot_n / rms_n)
    float a[kAttnResMaxSources], mx = -INFINITY;
#pragma unroll
    for (int n = 0; n < kAttnResMaxSources; ++n) {
        a[n] = n < p.M ? dot[n] * rsqrtf(ss[n] / (float)p.C + p.eps) : -INFINITY;
        mx = fmaxf(mx, a[n]);
    }
    float den = 0.f;
#pragma unroll
    for (int n = 0; n < kAttnResMaxSources; ++n) {
        a[n] = n < p.M ? __expf(a[n] - mx) : 0.f;
        den += a[n];
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int n = 0; n < kAttnResMaxSources; ++n) a[n] *= inv;

    const uint64_t last = evict_first_policy();
    uint4* o = reinterpret_cast<uint4*>(p.out + row);
#pragma unroll 2
    for (int ch = 0; ch < chunks; ++ch) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int n = 0; n < kAttnResMaxSources; ++n) {
            if (n < p.M) {
                float x[8];
                unpack8(ld_last(p.src[n] + row + ch * 256, last), x);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(a[n], x[i], acc[i]);
            }
        }
        o[ch * 32] = make_uint4(f2_to_bf2(acc[0], acc[1]), f2_to_bf2(acc[2], acc[3]),
                                f2_to_bf2(acc[4], acc[5]), f2_to_bf2(acc[6], acc[7]));
    }
}

}  // namespace

cudaError_t launch_attnres(const void* const* sources, int M, long long T, int C, const float* w,
                           float eps, void* out, cudaStream_t stream) {
    AttnResParams p{};
    for (int n = 0; n < M; ++n) p.src[n] = static_cast<const __nv_bfloat16*>(sources[n]);
    p.M = M;
    p.C = C;
    p.T = T;
    p.eps = eps;
    p.w = w;
    p.out = static_cast<__nv_bfloat16*>(out);
    const size_t smem = (size_t)C * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(attnres_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const long long blocks = (T + kArWarps - 1) / kArWarps;
    attnres_kernel<<<(unsigned)blocks, kArWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sla
