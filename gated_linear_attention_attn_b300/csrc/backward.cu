// Backward of the gated linear-attention layer.
//
// For one head, with num_i = qr_i^T S, den_i = phi(q_i) . z + eps and
// s_i = sigmoid(g_i), the gradients of L = sum(dO * o) are
//
//     a_i    = dO_i * s_i / den_i                 dg_i = dO_i * num_i / den_i * s_i (1 - s_i)
//     dden_i = -(a_i . num_i) / den_i
//     dS     = sum_i qr_i a_i^T                   dz   = sum_i dden_i phi(q_i)
//     dq_i   = [q_i > 0] (R_i^T (S a_i) + dden_i z)
//     dk_j   = [k_j > 0] (R_j^T (dS v_j) + dz)    dv_j = dS^T kr_j
//
// bf16 inputs: the contractions run on the tensor cores through the state and
// apply kernels, the elementwise terms in the apply kernel's epilogue:
//   1. state(k, v)                      S (bf16, as the forward uses it), z
//   2. apply, gate terms(q, g, dO; S)   num on the tensor cores; a, dg, dden in
//                                       the epilogue; dS partials from qr and a
//   3. apply, masked gradient(a; S, q)  S a on the tensor cores; dq in the
//                                       epilogue (mask of q, R^T, + dden z);
//                                       dz partials from the q tiles
//   4. dS merge                         dS (bf16, as S), dz
//   5. apply, masked gradient(v; dS, k) dS v; dk (mask of k, R^T, + dz)
//   6. apply, raw(k; dS)                dv = dS^T kr
// fp32 inputs: fp32 FMA kernels in three launches, each over (chunk of tokens,
// head): the state partials (simt_state_kernel); bwd_query_kernel (num, a, dg,
// dden, dq and the chunk's dS, dz); bwd_key_kernel (dk, dv).
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

constexpr int kBTile = 32;                          // tokens per tile
constexpr int kBThreads = 256;
constexpr int kBPartial = kHeadDim * kHeadDim + kHeadDim;
// S, S^T, z, then three [32][128] tiles and two [32] vectors
constexpr size_t kBSmem =
    (2 * kHeadDim * kHeadDim + kHeadDim + 3 * kBTile * kHeadDim + 2 * kBTile) * sizeof(float);

__device__ __forceinline__ float ld_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ void st_elem(float* p, float x) { *p = x; }

// Sums the C partials (chunk order) of a head into M ([m][n]), Mt ([n][m])
// and the vector part into vec, four elements per thread at a time so that
// four loads are in flight.
__device__ void sum_partials(const float* src, int C, float* M, float* Mt, float* vec) {
    for (int e0 = threadIdx.x; e0 < kBPartial; e0 += 4 * blockDim.x) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int cc = 0; cc < C; ++cc) {
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * blockDim.x;
                x[u] = e < kBPartial ? __ldcg(src + (size_t)cc * kBPartial + e) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] += x[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * blockDim.x;
            if (e < kHeadDim * kHeadDim) {
                M[e] = s[u];
                Mt[(e % kHeadDim) * kHeadDim + e / kHeadDim] = s[u];
            } else if (e < kBPartial) {
                vec[e - kHeadDim * kHeadDim] = s[u];
            }
        }
    }
}

// Loads rows [base, base + cnt) of a head into fp (ReLU) and fr (ReLU, then
// rotated); rows past cnt are zero.
template <typename T, bool ROPE>
__device__ void load_features(const T* x, int base, int cnt, RopeView rope, float* fp, float* fr) {
    for (int e = threadIdx.x; e < kBTile * kHeadDim; e += blockDim.x) {
        const int r = e / kHeadDim;
        const float xv = r < cnt ? ld_elem(x + (size_t)(base + r) * kHeadDim + e % kHeadDim) : 0.f;
        fp[e] = fmaxf(xv, 0.f);
        fr[e] = fp[e];
    }
    if (ROPE) {
        __syncthreads();
        const float2* cs = rope_pairs(rope);
        for (int e = threadIdx.x; e < cnt * kPairs; e += blockDim.x) {
            const int r = e / kPairs, p = e % kPairs;
            rotate_pair(fr[r * kHeadDim + 2 * p], fr[r * kHeadDim + 2 * p + 1],
                        __ldg(cs + (size_t)(base + r) * kPairs + p));
        }
    }
}

// A thread's eight columns of a [*][128] row: 4 tx .. 4 tx + 3 and
// 64 + 4 tx .. 64 + 4 tx + 3 (two whole pairs each; a warp's 16-byte loads of
// one row then fall in distinct banks).
__device__ __forceinline__ int col_of(int tx, int j) { return (j < 4 ? 0 : 64 - 4) + 4 * tx + j; }

// y[i][j] = sum_m X[(2 ty + i)][m] * M[m][col_of(tx, j)] for the two rows of this
// thread: X [32][128] and M [128][128] in shared memory.
__device__ __forceinline__ void rows_times(const float* X, const float* M, int ty, int tx,
                                           float (&y)[2][8]) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) y[i][j] = 0.f;
    const float* x0 = X + (2 * ty) * kHeadDim;
    const float* x1 = x0 + kHeadDim;
#pragma unroll 2
    for (int m = 0; m < kHeadDim; m += 4) {
        const float4 a0 = *reinterpret_cast<const float4*>(x0 + m);
        const float4 a1 = *reinterpret_cast<const float4*>(x1 + m);
        const float av0[4] = {a0.x, a0.y, a0.z, a0.w};
        const float av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float* row = M + (m + mm) * kHeadDim + 4 * tx;
            const float4 b0 = *reinterpret_cast<const float4*>(row);
            const float4 b1 = *reinterpret_cast<const float4*>(row + 64);
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                y[0][j] = fmaf(av0[mm], b[j], y[0][j]);
                y[1][j] = fmaf(av1[mm], b[j], y[1][j]);
            }
        }
    }
}

// y = R^T y on this thread's four pairs (columns col_of(tx, 0..7)) of row n.
template <bool ROPE>
__device__ __forceinline__ void unrotate8(float (&y)[8], const RopeView& rope, int n, int tx) {
    if (!ROPE) return;
    const float2* row = rope_pairs(rope) + (size_t)n * kPairs;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 cs = __ldg(row + col_of(tx, 2 * p) / 2);
        rotate_pair(y[2 * p], y[2 * p + 1], make_float2(cs.x, -cs.y));
    }
}

template <typename T, bool ROPE>
__global__ void __launch_bounds__(kBThreads)
bwd_query_kernel(const T* __restrict__ q, const T* __restrict__ g, const T* __restrict__ dout,
                 T* __restrict__ dq, T* __restrict__ dg, int N, int C, int chunk,
                 const float* __restrict__ state_partial, float* __restrict__ grad_partial,
                 float eps, RopeView rope) {
    extern __shared__ float sm[];
    float* S = sm;                                   // [m][n]
    float* St = S + kHeadDim * kHeadDim;             // [n][m]
    float* z = St + kHeadDim * kHeadDim;
    float* qp = z + kHeadDim;                        // [32][128] phi(q)
    float* qr = qp + kBTile * kHeadDim;              // [32][128] R phi(q)
    float* a = qr + kBTile * kHeadDim;               // [32][128] dL/dnum
    float* den = a + kBTile * kHeadDim;              // [32]
    float* dden = den + kBTile;                      // [32]
    const int bh = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    if (ROPE && !rope_table_ok(rope)) return;        // reported by the state partials
    const int ty = tid / 16, tx = tid % 16;
    const size_t head = (size_t)bh * N * kHeadDim;
    // the head's S, z, summed from the fp32 partials
    sum_partials(state_partial + (size_t)bh * C * kBPartial, C, S, St, z);

    float acc[8][8];                          // dS rows 8 ty.., columns col_of(tx, ..)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float dzacc = 0.f;                               // dz[tid] for tid < 128

    const int n0 = c * chunk, n1 = min(N, n0 + chunk);
    for (int base = n0; base < n1; base += kBTile) {
        const int cnt = min(kBTile, n1 - base);
        __syncthreads();
        load_features<T, ROPE>(q + head, base, cnt, rope, qp, qr);
        __syncthreads();
        {   // den_r = phi(q_r) . z + eps, one warp per row at a time
            const int warp = tid / 32, lane = tid % 32;
            for (int r = warp; r < kBTile; r += kBThreads / 32) {
                float s = 0.f;
                for (int col = lane; col < kHeadDim; col += 32) s = fmaf(qp[r * kHeadDim + col], z[col], s);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (lane == 0) den[r] = s + eps;
            }
        }
        __syncthreads();
        // num = qr S for rows 2 ty, 2 ty + 1 and this thread's columns
        float num[2][8];
        rows_times(qr, S, ty, tx, num);
        // a, dg and this thread's share of a . num
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = 2 * ty + i;
            float part = 0.f;
            if (r < cnt) {
                const size_t row = head + (size_t)(base + r) * kHeadDim;
                const float inv_den = 1.f / den[r];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = col_of(tx, j);
                    const float s = 1.f / (1.f + expf(-ld_elem(g + row + col)));
                    const float gd = ld_elem(dout + row + col);
                    const float av = gd * s * inv_den;
                    a[r * kHeadDim + col] = av;
                    st_elem(dg + row + col, gd * num[i][j] * inv_den * s * (1.f - s));
                    part = fmaf(av, num[i][j], part);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) a[r * kHeadDim + col_of(tx, j)] = 0.f;
            }
            // the 16 threads of a row are lanes 16 (ty & 1) .. + 15 of one warp
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (tx == 0) dden[r] = r < cnt ? -part / den[r] : 0.f;
        }
        __syncthreads();
        // dq = [q > 0] (R^T (S a) + dden z): S a is sum_n a[r][n] S[m][n] = sum_n a[r][n] St[n][m]
        {
            float y[2][8];
            rows_times(a, St, ty, tx, y);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = 2 * ty + i;
                if (r >= cnt) continue;
                unrotate8<ROPE>(y[i], rope, base + r, tx);
                const size_t row = head + (size_t)(base + r) * kHeadDim;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int col = col_of(tx, j);
                    const float v = qp[r * kHeadDim + col] > 0.f ? y[i][j] + dden[r] * z[col] : 0.f;
                    st_elem(dq + row + col, v);
                }
            }
        }
        // the tile's share of dS = sum_r qr_r a_r^T and dz = sum_r dden_r phi(q_r)
        for (int r = 0; r < cnt; ++r) {
            float x[8], w[8];
            const float4 x0 = *reinterpret_cast<const float4*>(qr + r * kHeadDim + ty * 8);
            const float4 x1 = *reinterpret_cast<const float4*>(qr + r * kHeadDim + ty * 8 + 4);
            const float4 w0 = *reinterpret_cast<const float4*>(a + r * kHeadDim + 4 * tx);
            const float4 w1 = *reinterpret_cast<const float4*>(a + r * kHeadDim + 64 + 4 * tx);
            x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
            x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
            w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
            w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(x[i], w[j], acc[i][j]);
        }
        if (tid < kHeadDim)
            for (int r = 0; r < cnt; ++r) dzacc = fmaf(dden[r], qp[r * kHeadDim + tid], dzacc);
    }
    float* dst = grad_partial + ((size_t)bh * C + c) * kBPartial;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(ty * 8 + i) * kHeadDim + col_of(tx, j)] = acc[i][j];
    if (tid < kHeadDim) dst[kHeadDim * kHeadDim + tid] = dzacc;
}

template <typename T, bool ROPE>
__global__ void __launch_bounds__(kBThreads)
bwd_key_kernel(const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ dk,
               T* __restrict__ dv, int N, int C, int chunk, const float* __restrict__ grad_partial,
               RopeView rope) {
    extern __shared__ float sm[];
    float* dS = sm;                                  // [m][n]
    float* dSt = dS + kHeadDim * kHeadDim;           // [n][m]
    float* dz = dSt + kHeadDim * kHeadDim;
    float* kp = dz + kHeadDim;                       // [32][128] phi(k)
    float* kr = kp + kBTile * kHeadDim;              // [32][128] R phi(k)
    float* vs = kr + kBTile * kHeadDim;              // [32][128] v
    const int bh = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    if (ROPE && !rope_table_ok(rope)) return;        // reported by the state partials
    const int ty = tid / 16, tx = tid % 16;
    const size_t head = (size_t)bh * N * kHeadDim;
    sum_partials(grad_partial + (size_t)bh * C * kBPartial, C, dS, dSt, dz);

    const int n0 = c * chunk, n1 = min(N, n0 + chunk);
    for (int base = n0; base < n1; base += kBTile) {
        const int cnt = min(kBTile, n1 - base);
        __syncthreads();
        load_features<T, ROPE>(k + head, base, cnt, rope, kp, kr);
        for (int e = tid; e < kBTile * kHeadDim; e += blockDim.x) {
            const int r = e / kHeadDim;
            vs[e] = r < cnt ? ld_elem(v + head + (size_t)(base + r) * kHeadDim + e % kHeadDim) : 0.f;
        }
        __syncthreads();
        // dS v_j = sum_n v[j][n] dS^T[n][m] (columns m); dS^T kr_j = sum_m kr[j][m] dS[m][n]
        // (columns n)
        float y[2][8], w[2][8];
        rows_times(vs, dSt, ty, tx, y);
        rows_times(kr, dS, ty, tx, w);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = 2 * ty + i;
            if (r >= cnt) continue;
            unrotate8<ROPE>(y[i], rope, base + r, tx);
            const size_t row = head + (size_t)(base + r) * kHeadDim;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = col_of(tx, j);
                st_elem(dk + row + col, kp[r * kHeadDim + col] > 0.f ? y[i][j] + dz[col] : 0.f);
                st_elem(dv + row + col, w[i][j]);
            }
        }
    }
}

// ------------------------------------------------ bf16, on the tensor cores

constexpr int kStateBytesB = kHeadDim * kHeadDim * 2 + kHeadDim * 4;   // bf16 S^T, then z

template <typename T>
cudaError_t launch_backward(const T* q, const T* k, const T* v, const T* g, const T* dout, T* dq,
                            T* dk, T* dv, T* dg, int B, int H, int N, const RopeView* rope,
                            float eps, float* workspace, int C, unsigned* status,
                            cudaStream_t stream) {
    const int BH = B * H;
    const int tiles = (N + kBTile - 1) / kBTile;
    const int chunk = ((tiles + C - 1) / C) * kBTile;
    const RopeView rv = rope ? *rope : RopeView{};
    float* state_partial = workspace;
    float* grad_partial = workspace + (size_t)BH * C * kBPartial;
    cudaError_t e = cudaSuccess;
    if ((e = launch_simt_state_partials(k, v, B, H, N, rope, state_partial, C, status,
                                        stream)) != cudaSuccess)
        return e;
    const dim3 grid(C, BH);
    if (rope) {
        cudaFuncSetAttribute(bwd_query_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBSmem);
        cudaFuncSetAttribute(bwd_key_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBSmem);
        bwd_query_kernel<T, true><<<grid, kBThreads, kBSmem, stream>>>(
            q, g, dout, dq, dg, N, C, chunk, state_partial, grad_partial, eps, rv);
        bwd_key_kernel<T, true><<<grid, kBThreads, kBSmem, stream>>>(k, v, dk, dv, N, C, chunk,
                                                                     grad_partial, rv);
    } else {
        cudaFuncSetAttribute(bwd_query_kernel<T, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBSmem);
        cudaFuncSetAttribute(bwd_key_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBSmem);
        bwd_query_kernel<T, false><<<grid, kBThreads, kBSmem, stream>>>(
            q, g, dout, dq, dg, N, C, chunk, state_partial, grad_partial, eps, rv);
        bwd_key_kernel<T, false><<<grid, kBThreads, kBSmem, stream>>>(k, v, dk, dv, N, C, chunk,
                                                                      grad_partial, rv);
    }
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_bytes(int BH, int C) {
    return 2 * (size_t)BH * C * kBPartial * sizeof(float);
}

static size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

size_t backward_bf16_workspace_bytes(int BH, int N, int num_sms) {
    const size_t tensor = (size_t)BH * N * kHeadDim * 2;
    return tc_state_workspace_bytes(BH, N, num_sms) + 2 * (size_t)BH * kStateBytesB + tensor +
           round_up((size_t)BH * N * sizeof(float)) + tc_apply_partial_bytes(BH, N, num_sms) +
           tc_apply_zpart_bytes(BH, N, num_sms) + 1024;
}

cudaError_t launch_backward_bf16(const void* q, const void* k, const void* v, const void* g,
                                 const void* dout, void* dq, void* dk, void* dv, void* dg, int B,
                                 int H, int N, const RopeView* rope, float eps, float* workspace,
                                 int num_sms, unsigned* status, cudaStream_t stream,
                                 const void* state) {
    const int BH = B * H;
    const size_t tensor = (size_t)BH * N * kHeadDim * 2;
    // workspace: the state kernel's, the two states, a ([rows][128] bf16), dden,
    // then the partials of dS and of dz
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    uint8_t* own_S = ws + tc_state_workspace_bytes(BH, N, num_sms);
    const void* S = state ? state : own_S;      // a given state is only read
    uint8_t* dS = own_S + (size_t)BH * kStateBytesB;
    uint8_t* A = dS + (size_t)BH * kStateBytesB;
    float* dden = reinterpret_cast<float*>(A + tensor);
    float* dspart = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dden) +
                                             round_up((size_t)BH * N * sizeof(float)));
    float* dzpart = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dspart) +
                                             tc_apply_partial_bytes(BH, N, num_sms));
    cudaError_t e;
    // Each launch after the first is a programmatic dependent of the one before:
    // its CTAs set up (and, where its tiles are inputs of the call, prefetch) as
    // the previous grid's CTAs leave their SMs.
    // (with a given state the gate terms are the call's first launch, and wait
    // for whatever ran before on the stream, as its tiles may come from there)
    if (!state &&
        (e = launch_tc_state(k, v, own_S, B, H, N, rope, ws, status, num_sms, stream)) !=
            cudaSuccess)
        return e;
    // num on the tensor cores, the gate terms in the apply kernel's epilogue (a, dg,
    // dden), and dS = sum qr a^T from the same tiles
    if ((e = launch_tc_apply(q, g, S, A, B, H, N, rope, eps, status, num_sms, stream,
                             kApplyTerms, dout, dg, dden, dspart, nullptr,
                             state ? kPdlNone : kPdlState)) != cudaSuccess)
        return e;
    // dq = [q > 0] (R^T (S a) + dden z), and dz = sum dden phi(q) from its q tiles
    // (a and dden come from the launch before: nothing of them is read before it
    // ends; the q tiles, inputs of the call, are prefetched)
    if ((e = launch_tc_apply(A, q, S, dq, B, H, N, rope, eps, status, num_sms, stream,
                             kApplyGrad, nullptr, nullptr, dden, nullptr, dzpart,
                             kPdlWaitAllButG)) != cudaSuccess)
        return e;
    if ((e = launch_tc_ds_merge(dspart, dzpart, dS, B, H, N, num_sms, stream, true)) !=
        cudaSuccess)
        return e;
    // dk = [k > 0] (R^T (dS v) + dz), dv = dS^T kr; v and k prefetched, dS waited for
    if ((e = launch_tc_apply(v, k, dS, dk, B, H, N, rope, eps, status, num_sms, stream,
                             kApplyGrad, nullptr, nullptr, nullptr, nullptr, nullptr,
                             kPdlState)) != cudaSuccess)
        return e;
    return launch_tc_apply(k, k, dS, dv, B, H, N, rope, eps, status, num_sms, stream, kApplyRaw,
                           nullptr, nullptr, nullptr, nullptr, nullptr, kPdlState);
}

cudaError_t launch_backward_f32(const float* q, const float* k, const float* v, const float* g,
                                const float* dout, float* dq, float* dk, float* dv, float* dg,
                                int B, int H, int N, const RopeView* rope, float eps,
                                float* workspace, int C, unsigned* status, cudaStream_t stream) {
    return launch_backward<float>(q, k, v, g, dout, dq, dk, dv, dg, B, H, N, rope, eps, workspace,
                                  C, status, stream);
}

}  // namespace sla
