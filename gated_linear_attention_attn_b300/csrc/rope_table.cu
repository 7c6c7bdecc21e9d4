// The 3D RoPE table: (cos, sin) of pos * base^(-2j/W) for each axis band.
//
// "Wan 3D rotary position embeddings" (SANA-Video 2.0, NVlabs/Sana
// docs/sana_video2.md, "Architecture") rotate the t, h and w bands of the
// head dimension by the token's frame, row and column index.  The table holds,
// after a header that describes it, every token's d/2 (cos, sin) pairs twice:
// as fp16 pairs, which the tensor-core kernels stream next to the token's row
// of q or k, and as fp32 pairs ([N][d/2][2]), which the fp32 kernels read.
// The header lets every kernel check the table against its call before it
// reads anything else.
#include <cuda_fp16.h>

#include "launch.h"

namespace sla {
namespace {

// The 64 header words (layout in common.cuh).
struct RopeHeader {
    uint32_t w[16];
};

RopeHeader make_header(int N, int d, int T, int Hs, int Ws, int dt, int dh, int dw, float base) {
    RopeHeader h{};
    h.w[kRopeHdrMagic] = kRopeMagic;
    h.w[kRopeHdrVersion] = kRopeVersion;
    h.w[kRopeHdrN] = (uint32_t)N;
    h.w[kRopeHdrD] = (uint32_t)d;
    h.w[kRopeHdrT] = (uint32_t)T;
    h.w[kRopeHdrHs] = (uint32_t)Hs;
    h.w[kRopeHdrWs] = (uint32_t)Ws;
    h.w[kRopeHdrDt] = (uint32_t)dt;
    h.w[kRopeHdrDh] = (uint32_t)dh;
    h.w[kRopeHdrDw] = (uint32_t)dw;
    uint32_t b;
    static_assert(sizeof(b) == sizeof(base), "fp32 base");
    __builtin_memcpy(&b, &base, sizeof(b));
    h.w[kRopeHdrBase] = b;
    h.w[kRopeHdrRows] = (uint32_t)kRopeHeaderWords;
    h.w[kRopeHdrPairs] = (uint32_t)(kRopeHeaderWords + (size_t)N * (d / 2));
    return h;
}

__device__ __forceinline__ void write_header(uint32_t* table, const RopeHeader& h) {
    if (blockIdx.x == 0 && threadIdx.x < kRopeHeaderWords)
        table[threadIdx.x] = threadIdx.x < 16 ? h.w[threadIdx.x] : 0u;
}

__device__ __forceinline__ uint32_t half2_bits(float c, float s) {
    const __half2 v = __floats2half2_rn(c, s);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// theta_j = base^(-2j/W) for pair j of a band of width W = 2 * pairs.
__device__ __forceinline__ double band_angle(double base, int pos, int j, int pairs) {
    return (double)pos * pow(base, -(double)j / (double)pairs);
}

// Entry (n, p): pair p of token n = (t*Hs + h)*Ws + w.  The pair's band gives
// the coordinate (t, h or w) and the ladder position j inside the band; the
// angle and its cosine and sine are taken in double precision, stored rounded
// to fp32, and the fp32 values rounded again to fp16.
__global__ void rope_fill_kernel(uint32_t* __restrict__ table, int T, int Hs, int Ws, int pt,
                                 int ph, int pw, double base, RopeHeader hdr) {
    write_header(table, hdr);
    const int P = pt + ph + pw;
    const int total = T * Hs * Ws * P;
    uint32_t* rows = table + kRopeHeaderWords;
    float2* pairs = reinterpret_cast<float2*>(rows + total);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += gridDim.x * blockDim.x) {
        const int n = e / P, p = e - n * P;
        const int hw = n / Ws, w = n - hw * Ws;
        const int t = hw / Hs, h = hw - t * Hs;
        int pos, j, band;
        if (p < pt) {
            pos = t, j = p, band = pt;
        } else if (p < pt + ph) {
            pos = h, j = p - pt, band = ph;
        } else {
            pos = w, j = p - pt - ph, band = pw;
        }
        double s, c;
        sincos(band_angle(base, pos, j, band), &s, &c);
        const float2 cs = make_float2((float)c, (float)s);
        pairs[e] = cs;
        rows[e] = half2_bits(cs.x, cs.y);
    }
}

// A table from caller-given fp32 pairs [N][P][2]: copied, and rounded to fp16.
__global__ void rope_from_pairs_kernel(uint32_t* __restrict__ table,
                                       const float2* __restrict__ src, int total,
                                       RopeHeader hdr) {
    write_header(table, hdr);
    uint32_t* rows = table + kRopeHeaderWords;
    float2* pairs = reinterpret_cast<float2*>(rows + total);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += gridDim.x * blockDim.x) {
        const float2 cs = src[e];
        pairs[e] = cs;
        rows[e] = half2_bits(cs.x, cs.y);
    }
}

int grid_for(long long total, int threads) {
    long long blocks = (total + threads - 1) / threads;
    return blocks > 4096 ? 4096 : (blocks < 1 ? 1 : (int)blocks);
}

}  // namespace

cudaError_t launch_rope_fill(float* table, int T, int Hs, int Ws, int dt, int dh, int dw,
                             float base, cudaStream_t stream) {
    const int N = T * Hs * Ws, d = dt + dh + dw;
    const RopeHeader hdr = make_header(N, d, T, Hs, Ws, dt, dh, dw, base);
    const int threads = 256;
    rope_fill_kernel<<<grid_for((long long)N * (d / 2), threads), threads, 0, stream>>>(
        reinterpret_cast<uint32_t*>(table), T, Hs, Ws, dt / 2, dh / 2, dw / 2, (double)base, hdr);
    return cudaGetLastError();
}

cudaError_t launch_rope_from_pairs(float* table, const float* pairs, int N, int d,
                                   cudaStream_t stream) {
    const RopeHeader hdr = make_header(N, d, 0, 0, 0, 0, 0, 0, 0.f);
    const int threads = 256;
    const int total = N * (d / 2);
    rope_from_pairs_kernel<<<grid_for(total, threads), threads, 0, stream>>>(
        reinterpret_cast<uint32_t*>(table), reinterpret_cast<const float2*>(pairs), total, hdr);
    return cudaGetLastError();
}

}  // namespace sla
