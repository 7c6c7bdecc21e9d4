// The 3D RoPE table: (cos, sin) of pos * base^(-2j/W) for each axis band.
//
// "Wan 3D rotary position embeddings" (SANA-Video 2.0, NVlabs/Sana
// docs/sana_video2.md, "Architecture") rotate the t, h and w bands of the
// head dimension by the token's frame, row and column index.  The angles of a
// band depend on one coordinate only, so the table holds one short row per
// coordinate value instead of one row per token.
#include "launch.h"

namespace sla {
namespace {

__global__ void rope_fill_kernel(float2* __restrict__ table, int T, int Hs, int Ws, int pt,
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
        // band width W = 2 * pairs; theta_j = base^(-2j/W) = base^(-j/pairs)
        const double theta = pow(base, -(double)j / (double)pairs);
        double s, c;
        sincos((double)pos * theta, &s, &c);
        table[e] = make_float2((float)c, (float)s);
    }
}

}  // namespace

cudaError_t launch_rope_fill(float* table, int T, int Hs, int Ws, int dt, int dh, int dw,
                             float base, cudaStream_t stream) {
    const int total = T * (dt / 2) + Hs * (dh / 2) + Ws * (dw / 2);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    int blocks = (total + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    rope_fill_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<float2*>(table), T, Hs,
                                                      Ws, dt / 2, dh / 2, dw / 2, (double)base);
    return cudaGetLastError();
}

}  // namespace sla
