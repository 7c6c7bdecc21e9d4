// fp32 path of the linear-attention forward: plain SIMT FFMA kernels.
//
// fp32 tensors need fp32 arithmetic end to end (a tf32 tensor-core product
// would be ~1e-3 off), so this path does not use the tensor cores.  It runs
// in two launches:
//   simt_state_kernel  grid (C, B*H): chunk c of a head forms the partial
//                      S_c = sum_j R_j phi(k_j) v_j^T and z_c = sum_j phi(k_j)
//                      over its tokens, written to the workspace;
//   simt_apply_kernel  grid (ceil(N/32), B*H): sums the C partials of its
//                      head, then evaluates o_i for 32 tokens.
#include "common.cuh"
#include "launch.h"

namespace sla {
namespace {

constexpr int kSimtTile = 32;                       // tokens per smem tile
constexpr int kPartialFloats = kHeadDim * kHeadDim + kHeadDim;

__device__ __forceinline__ float load_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ void store_elem(float* p, float x) { *p = x; }

template <typename T, bool ROPE>
__global__ void __launch_bounds__(256)
simt_state_kernel(const T* __restrict__ k, const T* __restrict__ v, int N, int C,
                  int chunk, RopeView rope, float* __restrict__ partial, unsigned* rope_status) {
    __shared__ float ks[kSimtTile][kHeadDim];
    __shared__ float vs[kSimtTile][kHeadDim];
    const int bh = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    if (ROPE && !rope_table_ok(rope)) {        // the whole block leaves; nothing is read
        if (tid == 0 && c == 0 && bh == 0) raise_status(rope_status, kStatusBadTable);
        return;
    }
    const float2* cs = ROPE ? rope_pairs(rope) : nullptr;
    const int ty = tid / 16, tx = tid % 16;
    const size_t head = (size_t)bh * N * kHeadDim;
    const int n0 = c * chunk;
    const int n1 = min(N, n0 + chunk);

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float zacc = 0.f;

    for (int base = n0; base < n1; base += kSimtTile) {
        const int cnt = min(kSimtTile, n1 - base);
        for (int e = tid; e < kSimtTile * kHeadDim; e += blockDim.x) {
            const int r = e / kHeadDim, col = e % kHeadDim;
            float kv = 0.f, vv = 0.f;
            if (r < cnt) {
                kv = fmaxf(load_elem(k + head + (size_t)(base + r) * kHeadDim + col), 0.f);
                vv = load_elem(v + head + (size_t)(base + r) * kHeadDim + col);
            }
            ks[r][col] = kv;
            vs[r][col] = vv;
        }
        __syncthreads();
        if (tid < kHeadDim) {
            for (int r = 0; r < cnt; ++r) zacc += ks[r][tid];   // unrotated phi(k)
        }
        if (ROPE) {
            __syncthreads();
            for (int e = tid; e < cnt * kPairs; e += blockDim.x) {
                const int r = e / kPairs, p = e % kPairs;
                rotate_pair(ks[r][2 * p], ks[r][2 * p + 1],
                            __ldg(cs + (size_t)(base + r) * kPairs + p));
            }
        }
        __syncthreads();
        for (int j = 0; j < cnt; ++j) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a[i] = ks[j][ty * 8 + i];
                b[i] = vs[j][tx * 8 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
        }
        __syncthreads();
    }

    float* dst = partial + ((size_t)bh * C + c) * kPartialFloats;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            dst[(ty * 8 + i) * kHeadDim + tx * 8 + jj] = acc[i][jj];
    if (tid < kHeadDim) dst[kHeadDim * kHeadDim + tid] = zacc;
}

template <typename T, bool ROPE>
__global__ void __launch_bounds__(256)
simt_apply_kernel(const T* __restrict__ q, const T* __restrict__ g,
                  T* __restrict__ out, int N, int C, const float* __restrict__ partial,
                  float eps, RopeView rope) {
    if (ROPE && !rope_table_ok(rope)) return;   // reported by the state kernel
    extern __shared__ float smem[];
    float* S = smem;                                 // [128][128]
    float* z = S + kHeadDim * kHeadDim;              // [128]
    float* qs = z + kHeadDim;                        // [32][128]
    float* den = qs + kSimtTile * kHeadDim;          // [32]
    const int bh = blockIdx.y, tid = threadIdx.x;
    const int base = blockIdx.x * kSimtTile;
    const int cnt = min(kSimtTile, N - base);
    const size_t head = (size_t)bh * N * kHeadDim;

    // The head's state: the C partials summed in chunk order, four elements per
    // thread at a time so that four loads are in flight.
    const float* src = partial + (size_t)bh * C * kPartialFloats;
    for (int e0 = tid; e0 < kPartialFloats; e0 += 4 * blockDim.x) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cc = 0; cc < C; ++cc) {
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * blockDim.x;
                x[u] = e < kPartialFloats ? src[(size_t)cc * kPartialFloats + e] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] += x[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (e0 + u * blockDim.x < kPartialFloats) smem[e0 + u * blockDim.x] = s[u];
    }
    for (int e = tid; e < kSimtTile * kHeadDim; e += blockDim.x) {
        const int r = e / kHeadDim, col = e % kHeadDim;
        qs[e] = r < cnt ? fmaxf(load_elem(q + head + (size_t)(base + r) * kHeadDim + col), 0.f)
                        : 0.f;
    }
    __syncthreads();
    // den_r = phi(q_r) . z + eps on the unrotated features: one warp per 4 rows
    {
        const int warp = tid / 32, lane = tid % 32;
        for (int r = warp; r < kSimtTile; r += blockDim.x / 32) {
            float s = 0.f;
            for (int col = lane; col < kHeadDim; col += 32) s = fmaf(qs[r * kHeadDim + col], z[col], s);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) den[r] = s + eps;
        }
    }
    if (ROPE) {
        __syncthreads();
        for (int e = tid; e < cnt * kPairs; e += blockDim.x) {
            const int r = e / kPairs, p = e % kPairs;
            rotate_pair(qs[r * kHeadDim + 2 * p], qs[r * kHeadDim + 2 * p + 1],
                        __ldg(rope_pairs(rope) + (size_t)(base + r) * kPairs + p));
        }
    }
    __syncthreads();

    const int ty = tid / 16, tx = tid % 16;          // rows 2ty, 2ty+1; cols 8tx..8tx+7
    float acc[2][8];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int m = 0; m < kHeadDim; ++m) {
        const float a0 = qs[(2 * ty) * kHeadDim + m];
        const float a1 = qs[(2 * ty + 1) * kHeadDim + m];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float b = S[m * kHeadDim + tx * 8 + j];
            acc[0][j] = fmaf(a0, b, acc[0][j]);
            acc[1][j] = fmaf(a1, b, acc[1][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = 2 * ty + i;
        if (r >= cnt) continue;
        const size_t row = head + (size_t)(base + r) * kHeadDim;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = tx * 8 + j;
            const float gate = 1.f / (1.f + expf(-load_elem(g + row + col)));
            store_elem(out + row + col, gate * (acc[i][j] / den[r]));
        }
    }
}

}  // namespace

size_t simt_workspace_bytes(int BH, int C) {
    return (size_t)BH * C * kPartialFloats * sizeof(float);
}

int simt_chunks(int BH, int N, int num_sms) {
    const int tiles = (N + kSimtTile - 1) / kSimtTile;
    int C = (2 * num_sms + BH - 1) / BH;
    // every apply block sums all C partials of its head: keep at least four
    // tiles per chunk so that this sum stays short
    if (C > (tiles + 3) / 4) C = (tiles + 3) / 4;
    if (C < 1) C = 1;
    return C;
}

template <typename T>
static cudaError_t launch_simt(const T* q, const T* k, const T* v, const T* g, T* out, int B,
                               int H, int N, const RopeView* rope, float eps, float* workspace,
                               int C, unsigned* status, cudaStream_t stream) {
    const int BH = B * H;
    const int tiles = (N + kSimtTile - 1) / kSimtTile;
    const int chunk = ((tiles + C - 1) / C) * kSimtTile;
    const RopeView rv = rope ? *rope : RopeView{};
    const size_t apply_smem =
        (kPartialFloats + kSimtTile * kHeadDim + kSimtTile) * sizeof(float);
    dim3 gs(C, BH), ga(tiles, BH);
    if (rope) {
        cudaFuncSetAttribute(simt_apply_kernel<T, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)apply_smem);
        simt_state_kernel<T, true><<<gs, 256, 0, stream>>>(k, v, N, C, chunk, rv, workspace,
                                                            status);
        simt_apply_kernel<T, true><<<ga, 256, apply_smem, stream>>>(q, g, out, N, C, workspace,
                                                                     eps, rv);
    } else {
        cudaFuncSetAttribute(simt_apply_kernel<T, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)apply_smem);
        simt_state_kernel<T, false><<<gs, 256, 0, stream>>>(k, v, N, C, chunk, rv, workspace,
                                                             status);
        simt_apply_kernel<T, false><<<ga, 256, apply_smem, stream>>>(q, g, out, N, C,
                                                                      workspace, eps, rv);
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_state_partials(const T* k, const T* v, int B, int H, int N,
                                         const RopeView* rope, float* partial, int C,
                                         unsigned* status, cudaStream_t stream) {
    const int tiles = (N + kSimtTile - 1) / kSimtTile;
    const int chunk = ((tiles + C - 1) / C) * kSimtTile;
    const RopeView rv = rope ? *rope : RopeView{};
    const dim3 gs(C, B * H);
    if (rope)
        simt_state_kernel<T, true><<<gs, 256, 0, stream>>>(k, v, N, C, chunk, rv, partial,
                                                            status);
    else
        simt_state_kernel<T, false><<<gs, 256, 0, stream>>>(k, v, N, C, chunk, rv, partial,
                                                             status);
    return cudaGetLastError();
}

cudaError_t launch_simt_state_partials(const float* k, const float* v, int B, int H, int N,
                                       const RopeView* rope, float* partial, int C,
                                       unsigned* status, cudaStream_t stream) {
    return launch_state_partials<float>(k, v, B, H, N, rope, partial, C, status, stream);
}

cudaError_t launch_simt_f32(const float* q, const float* k, const float* v, const float* g,
                            float* out, int B, int H, int N, const RopeView* rope, float eps,
                            float* workspace, int C, unsigned* status, cudaStream_t stream) {
    return launch_simt<float>(q, k, v, g, out, B, H, N, rope, eps, workspace, C, status, stream);
}

}  // namespace sla
