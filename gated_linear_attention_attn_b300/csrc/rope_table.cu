// The 3D RoPE table: (cos, sin) of pos * base^(-2j/W) for each axis band.
//
// "Wan 3D rotary position embeddings" (SANA-Video 2.0, NVlabs/Sana
// docs/sana_video2.md, "Architecture") rotate the t, h and w bands of the
// head dimension by the token's frame, row and column index.  The angles of a
// band depend on one coordinate only, so the first part of the table holds
// one short fp32 row per coordinate value (read by the fp32 kernels); the
// second part holds, for every token, all d/2 pairs as fp16 (cos, sin) copied
// from those rows, so that the tensor-core kernels stream a token's rotation
// with its row of q or k instead of gathering it pair by pair.
#include <cuda_fp16.h>

#include "launch.h"

namespace sla {
namespace {

// theta_j = base^(-2j/W) for pair j of a band of width W = 2 * pairs.
__device__ __forceinline__ double band_angle(double base, int pos, int j, int pairs) {
    return (double)pos * pow(base, -(double)j / (double)pairs);
}

__global__ void rope_axes_kernel(float2* __restrict__ table, int T, int Hs, int Ws, int pt,
                                 int ph, int pw, double base) {
    const int total = T * pt + Hs * ph + Ws * pw;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += gridDim.x * blockDim.x) {
        int pos, j, pairs;
        if (e < T * pt) {
            pairs = pt;
            pos = e / pt;
            j = e - pos * pt;
        } else if (e < T * pt + Hs * ph) {
            const int f = e - T * pt;
            pairs = ph;
            pos = f / ph;
            j = f - pos * ph;
        } else {
            const int f = e - T * pt - Hs * ph;
            pairs = pw;
            pos = f / pw;
            j = f - pos * pw;
        }
        double s, c;
        sincos(band_angle(base, pos, j, pairs), &s, &c);
        table[e] = make_float2((float)c, (float)s);
    }
}

// Entry (n, p): pair p of token n = (t*Hs + h)*Ws + w, copied from the axis
// rows (written just before on the same stream) and rounded to fp16.
__global__ void rope_tokens_kernel(uint32_t* __restrict__ rows, const float2* __restrict__ axes,
                                   int T, int Hs, int Ws, int pt, int ph, int pw) {
    const int P = pt + ph + pw;
    const int total = T * Hs * Ws * P;
    const float2* tab_h = axes + T * pt;
    const float2* tab_w = tab_h + Hs * ph;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += gridDim.x * blockDim.x) {
        const int n = e / P, p = e - n * P;
        const int hw = n / Ws, w = n - hw * Ws;
        const int t = hw / Hs, h = hw - t * Hs;
        float2 cs;
        if (p < pt)
            cs = axes[t * pt + p];
        else if (p < pt + ph)
            cs = tab_h[h * ph + (p - pt)];
        else
            cs = tab_w[w * pw + (p - pt - ph)];
        const __half2 v = __floats2half2_rn(cs.x, cs.y);
        rows[e] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

int grid_for(int total, int threads) {
    int blocks = (total + threads - 1) / threads;
    return blocks > 4096 ? 4096 : (blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_rope_fill(float* table, int T, int Hs, int Ws, int dt, int dh, int dw,
                             float base, cudaStream_t stream) {
    const int pt = dt / 2, ph = dh / 2, pw = dw / 2;
    const int axes = T * pt + Hs * ph + Ws * pw;
    const int tokens = T * Hs * Ws * (pt + ph + pw);
    const int threads = 256;
    if (axes > 0)
        rope_axes_kernel<<<grid_for(axes, threads), threads, 0, stream>>>(
            reinterpret_cast<float2*>(table), T, Hs, Ws, pt, ph, pw, (double)base);
    if (tokens > 0) {
        uint32_t* rows = reinterpret_cast<uint32_t*>(table) +
                         rope_tok_offset_words(T, Hs, Ws, dt, dh, dw);
        rope_tokens_kernel<<<grid_for(tokens, threads), threads, 0, stream>>>(
            rows, reinterpret_cast<const float2*>(table), T, Hs, Ws, pt, ph, pw);
    }
    return cudaGetLastError();
}

}  // namespace sla
