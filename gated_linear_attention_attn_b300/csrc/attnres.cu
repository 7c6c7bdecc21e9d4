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
// HBM-bound: every summary row is read once and x written once.  Each CTA
// works through its tokens (token blockIdx.x + k * gridDim.x) with a ring of
// 2 to 6 token slots in shared memory (about 70 KB, so several CTAs share an SM):
// one thread keeps bulk copies of the next tokens' M rows in flight
// (cp.async.bulk, completion counted on the slot's mbarrier).  Per token,
// thread i takes the 16-byte piece i of every row, the CTA reduces w . s_n
// and s_n . s_n (warp shuffles, then shared memory, one barrier), every warp
// forms the softmax, and thread i writes its piece of x from the rows it kept
// in registers (fp32 in CTAs of up to 384 threads, bf16 above that while they
// fit), else reading them again.
// Earlier forms measured slower: re-reading the rows from L2 in a second pass
// (the rows of the tokens in flight overflow L2 before the second read), and
// register prefetching one token ahead (too few bytes in flight).
#include <map>
#include <mutex>
#include <tuple>

#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

using namespace ptx;

constexpr int kArMaxThreads = 512;
constexpr int kArStages = 6;                // token slots: 2 .. 6, as many as fit the budget
// Per CTA: small rings and more CTAs per SM measured faster than deep rings
// (5B shape, 20 KB token slots: three slots and three CTAs per SM 209 us,
// five slots and two CTAs 225 us); a 40 KB slot (14B shape) still gets two.
constexpr size_t kArSmemBudget = 70 * 1024;

struct AttnResParams {
    const __nv_bfloat16* src[kAttnResMaxSources];
    int M;
    int C;                                  // a multiple of 256, at most 4096
    long long T;
    float eps;
    const float* w;
    __nv_bfloat16* out;
    unsigned* status;
    int stages;                             // token slots in shared memory, 1 .. kArStages
};

int attnres_stages(int M, int C) {
    const size_t slot = (size_t)M * C * 2;
    const size_t fit = kArSmemBudget / slot;
    return fit >= (size_t)kArStages ? kArStages : fit < 2 ? 2 : (int)fit;
}

// Sums P values over the 32 lanes of a warp with P - 1 + 5 - log2(P)
// shuffles instead of 5 P: each round halves the values a lane keeps.  On
// return v[0] of lane l holds the warp sum of value l >> (5 - log2 P).
template <int P>
__device__ __forceinline__ void warp_sum_transposed(float (&v)[P], int lane) {
    static_assert(P >= 1 && P <= 32 && (P & (P - 1)) == 0, "P a power of two up to 32");
    int off = 16;
#pragma unroll
    for (int width = P; width > 1; width >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < width / 2; ++i) {
            const float send = upper ? v[i] : v[i + width / 2];
            const float keep = upper ? v[i + width / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
}

template <int M>
struct PartCount {                          // 2 M rounded up to a power of two
    static constexpr int value = M <= 1 ? 2 : M <= 2 ? 4 : M <= 4 ? 8 : 16;
};

// How a thread holds its pieces of the token's rows between the reduction
// and the output.
constexpr int kArReread = 0;                // read again from shared memory
constexpr int kArKeepF32 = 1;               // in registers as fp32 (CTAs of <= 384 threads)
constexpr int kArKeepBf16 = 2;              // in registers as bf16: 4 words a row, so two
                                            // CTAs of 512 threads fit an SM (64 registers)

// blockDim.x * 8 == C: thread i owns columns 8i .. 8i + 7 of every row.
// Kept rows free their slot at the token's barrier, so the next fetch into
// it is issued one token earlier than when the rows are read again.
template <int M, int HOLD>
__global__ void __launch_bounds__(kArMaxThreads, HOLD == kArKeepBf16 ? 2 : 1)
attnres_kernel(AttnResParams p) {
    constexpr bool KEEP = HOLD != kArReread;
    constexpr int P = PartCount<M>::value;
    constexpr int kShift = P == 2 ? 4 : P == 4 ? 3 : P == 8 ? 2 : 1;   // 5 - log2 P
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float red[2][kArMaxThreads / 32][P];
    __shared__ uint64_t full[kArStages];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t row_bytes = (uint32_t)p.C * 2;
    const uint32_t slot_bytes = (uint32_t)M * row_bytes;
    const long long mine = blockIdx.x < p.T ? (p.T - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int S = p.stages;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto fetch = [&](long long k) {          // token k of this CTA into slot k % S
        const int s = (int)(k % S);
        const size_t off = (size_t)(blockIdx.x + k * gridDim.x) * p.C;
        mbar_arrive_expect_tx(&full[s], slot_bytes);
#pragma unroll
        for (int n = 0; n < M; ++n)
            bulk_load(smem + (size_t)s * slot_bytes + (size_t)n * row_bytes, p.src[n] + off,
                      row_bytes, &full[s]);
    };
    if (tid == 0)
        for (long long k = 0; k < mine && k < S; ++k) fetch(k);
    // this thread's eight query weights; kArKeepBf16 reads them (from L1) for
    // every token instead of holding them, to stay within 64 registers
    auto load_w = [&](float2 (&wv)[4]) {
        const float4* w4 = reinterpret_cast<const float4*>(p.w + (size_t)tid * 8);
        const float4 a = __ldg(w4), b = __ldg(w4 + 1);
        wv[0] = make_float2(a.x, a.y);
        wv[1] = make_float2(a.z, a.w);
        wv[2] = make_float2(b.x, b.y);
        wv[3] = make_float2(b.z, b.w);
    };
    float2 wheld[4];
    if (HOLD != kArKeepBf16) load_w(wheld);
    const float inv_c = 1.f / (float)p.C;
    long long k = 0;
    for (; k < mine; ++k) {
        const int s = (int)(k % S), buf = (int)(k & 1);
        float2 wv[4];
        if (HOLD == kArKeepBf16) {
            load_w(wv);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] = wheld[i];
        }
        const bool ok = mbar_wait(&full[s], (uint32_t)(k / S) & 1u, &abort_flag, p.status);
        const uint32_t slot = smem_u32(smem + (size_t)s * slot_bytes) + tid * 16;
        float2 x[M][4];                          // kept to the output when kArKeepF32
        uint4 raw[M];                            // kept to the output when kArKeepBf16
        float part[P];
#pragma unroll
        for (int n = 0; n < M; ++n) {
            const uint4 u = lds128(slot + n * row_bytes);
            if (HOLD == kArKeepBf16) raw[n] = u;
            x[n][0] = bf2_to_f2(u.x);
            x[n][1] = bf2_to_f2(u.y);
            x[n][2] = bf2_to_f2(u.z);
            x[n][3] = bf2_to_f2(u.w);
            float2 d = mul2(x[n][0], wv[0]), q = mul2(x[n][0], x[n][0]);
#pragma unroll
            for (int i = 1; i < 4; ++i) {
                d = fma2(x[n][i], wv[i], d);
                q = fma2(x[n][i], x[n][i], q);
            }
            part[2 * n] = d.x + d.y;
            part[2 * n + 1] = q.x + q.y;
        }
#pragma unroll
        for (int i = 2 * M; i < P; ++i) part[i] = 0.f;
        warp_sum_transposed<P>(part, lane);
        if ((lane & ((1 << kShift) - 1)) == 0) red[buf][wid][lane >> kShift] = part[0];
        // one barrier per token: the warps' partials are in, and every thread
        // learns whether any wait gave up (then nothing of this token is
        // stored).  A slot is free once its rows are read for the last time:
        // this token's slot now when KEEP, else the previous token's.
        if (__syncthreads_or(!ok)) break;
        if (KEEP) {
            if (tid == 0 && k + S < mine) fetch(k + S);
        } else {
            if (tid == 0 && k >= 1 && k - 1 + S < mine) fetch(k - 1 + S);
        }
        // every warp: lane i < P sums value i over the warps; lanes 2n, 2n + 1
        // hold w . s_n and s_n . s_n; a_n = softmax_n(dot_n / rms_n).
        // red[buf] is next written two tokens later, after the next barrier.
        float v = 0.f;
        if (lane < P)
            for (int w = 0; w < nwarps; ++w) v += red[buf][w][lane];
        const float q = __shfl_down_sync(0xffffffffu, v, 1);
        const float logit = v * rsqrtf(q * inv_c + p.eps);
        float a[M], mx = -INFINITY;
#pragma unroll
        for (int n = 0; n < M; ++n) {
            a[n] = __shfl_sync(0xffffffffu, logit, 2 * n);
            mx = fmaxf(mx, a[n]);
        }
        float den = 0.f;
#pragma unroll
        for (int n = 0; n < M; ++n) {
            a[n] = __expf(a[n] - mx);
            den += a[n];
        }
        const float inv = 1.f / den;
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int n = 0; n < M; ++n) {
            if (HOLD != kArKeepF32) {            // the rows again: from shared memory or bf16
                const uint4 u = HOLD == kArKeepBf16 ? raw[n] : lds128(slot + n * row_bytes);
                x[n][0] = bf2_to_f2(u.x);
                x[n][1] = bf2_to_f2(u.y);
                x[n][2] = bf2_to_f2(u.z);
                x[n][3] = bf2_to_f2(u.w);
            }
            const float an = a[n] * inv;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fma2(make_float2(an, an), x[n][i], acc[i]);
        }
        const size_t t = (size_t)(blockIdx.x + k * gridDim.x);
        *reinterpret_cast<uint4*>(p.out + t * p.C + (size_t)tid * 8) =
            make_uint4(f2_to_bf2(acc[0].x, acc[0].y), f2_to_bf2(acc[1].x, acc[1].y),
                       f2_to_bf2(acc[2].x, acc[2].y), f2_to_bf2(acc[3].x, acc[3].y));
    }
    if (tid == 0 && k < mine) {
        // gave up at token k: tokens k .. k + S - 1 (KEEP) or k .. k + S - 2
        // (k .. S - 1 when k is 0) were issued and may be in flight; they land
        // before the CTA exits
        const long long last = KEEP || k == 0 ? k + S - 1 : k + S - 2;
        for (long long j = k; j <= last && j < mine; ++j)
            mbar_wait_drain(&full[j % S], (uint32_t)(j / S) & 1u);
    }
}

}  // namespace

cudaError_t launch_attnres(const void* const* sources, int M, long long T, int C, const float* w,
                           float eps, void* out, unsigned* status, cudaStream_t stream) {
    AttnResParams p{};
    for (int n = 0; n < M; ++n) p.src[n] = static_cast<const __nv_bfloat16*>(sources[n]);
    p.M = M;
    p.C = C;
    p.T = T;
    p.eps = eps;
    p.w = w;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.status = status;
    p.stages = attnres_stages(M, C);
    const int threads = C / 8;                      // one 16-byte piece of a row each
    if (threads % 32 != 0 || threads > kArMaxThreads || p.stages < 1) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)p.stages * M * C * 2;
    // the grid (SMs x resident CTAs) per (device, kernel, threads, shared memory), found once:
    // later calls, also those inside a stream capture, make no attribute or occupancy calls.
    // The kernel's dynamic shared memory limit is raised to the device's whole opt-in
    // amount the first time, so that every later size (any C) launches without a call.
    auto launch = [&](auto kernel) -> cudaError_t {
        static std::mutex mu;
        static std::map<std::tuple<int, const void*, int, size_t>, long long> grids;
        long long blocks = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            const auto key = std::make_tuple(dev, reinterpret_cast<const void*>(kernel), threads,
                                             smem);
            auto it = grids.find(key);
            if (it == grids.end()) {
                int sms = 0, per_sm = 0;
                cudaError_t r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                cudaFuncAttributes fa{};
                int optin = 0;
                if (r == cudaSuccess) r = cudaFuncGetAttributes(&fa, kernel);
                if (r == cudaSuccess)
                    r = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                               dev);
                if (r == cudaSuccess)
                    r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             optin - (int)fa.sharedSizeBytes);
                if (r == cudaSuccess)
                    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads,
                                                                      smem);
                if (r != cudaSuccess) return r;
                it = grids.emplace(key, (long long)sms * (per_sm > 0 ? per_sm : 1)).first;
            }
            blocks = it->second;
        }
        if (blocks > T) blocks = T;
        kernel<<<(unsigned)blocks, threads, smem, stream>>>(p);
        return cudaGetLastError();
    };
    // rows held as fp32 up to 384 threads; above, as bf16 while that fits 64
    // registers without spilling much (M <= 5), else read again
    const int hold = threads <= 384 ? kArKeepF32 : M <= 5 ? kArKeepBf16 : kArReread;
    switch (M * 4 + hold) {
        case 5: return launch(attnres_kernel<1, kArKeepF32>);
        case 6: return launch(attnres_kernel<1, kArKeepBf16>);
        case 9: return launch(attnres_kernel<2, kArKeepF32>);
        case 10: return launch(attnres_kernel<2, kArKeepBf16>);
        case 13: return launch(attnres_kernel<3, kArKeepF32>);
        case 14: return launch(attnres_kernel<3, kArKeepBf16>);
        case 17: return launch(attnres_kernel<4, kArKeepF32>);
        case 18: return launch(attnres_kernel<4, kArKeepBf16>);
        case 21: return launch(attnres_kernel<5, kArKeepF32>);
        case 22: return launch(attnres_kernel<5, kArKeepBf16>);
        case 24: return launch(attnres_kernel<6, kArReread>);
        case 25: return launch(attnres_kernel<6, kArKeepF32>);
        case 28: return launch(attnres_kernel<7, kArReread>);
        case 29: return launch(attnres_kernel<7, kArKeepF32>);
        case 32: return launch(attnres_kernel<8, kArReread>);
        case 33: return launch(attnres_kernel<8, kArKeepF32>);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sla
