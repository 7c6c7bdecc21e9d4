// Shared pieces of the bf16 tensor-core kernels (tc_forward.cu, backward.cu):
// tile geometry, the stream-K split, the feature map, RoPE and gate helpers
// on 16-byte chunks, the per-head contributor counters, and the TMA tensor
// maps of [heads][N][128] bf16 tensors and of the per-token RoPE rows.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace tc {

using namespace ptx;

constexpr int kRowBytes = kHeadDim * 2;                          // one bf16 token row: 256 B
// A partial slot: S^T [128][128] fp32, then z [128] fp32.
constexpr int kPartialFloats = kHeadDim * kHeadDim + kHeadDim;
constexpr int kStateSBytes = kHeadDim * kHeadDim * 2;            // S^T bf16: 32 KB
constexpr int kStateBytes = kStateSBytes + kHeadDim * 4;         // + z fp32: 33280 B
constexpr int kStateHalf = kStateSBytes / 2;                     // one 64-column half

// ---- state kernel geometry
constexpr int kStTok = 64;                        // tokens per tile
constexpr int kStHalf = kStTok * 128;             // one 64-column box: 8 KB
constexpr int kStTile = 2 * kStHalf;              // one tensor tile: 16 KB
constexpr int kStRing = 6 * 2 * kStTile;          // the stage ring: 192 KB
constexpr int kStXWarps = 8;                      // transform warps
constexpr int kStFWarps = 4;                      // flush + merge warps
constexpr int kStXThreads = 32 * kStXWarps;
constexpr int kStThreads = 32 * (2 + kStXWarps + kStFWarps);   // + TMA warp, MMA warp
constexpr int kStTmemCols = 256;                  // two 128-column accumulators
constexpr int kStRowsPerThread = kStTok * 16 / kStXThreads;   // 4

// ---- apply kernel geometry
constexpr int kApTok = 128;
constexpr int kApHalf = kApTok * 128;             // 16 KB
constexpr int kApTile = 2 * kApHalf;              // 32 KB
constexpr int kApQStages = 3;                     // Q ring: a slot is free once the MMA read it
constexpr int kApGStages = 3;                     // G ring: a slot is free once o is stored
constexpr int kApDSlots = 4;                      // den of the tiles between transform and epilogue

// A state stage holds one tile of K and of V and, with RoPE, the tile's rows
// of the per-token RoPE table (256 bytes per token, the size of a tensor
// row); the ring has the same size either way, so RoPE trades stages for the
// table rows.  The apply kernel streams Q and G in separate rings, so a Q slot
// turns over as soon as the MMA has read it; its transform warps read their
// RoPE rows straight from global memory (L2), one tile ahead.
template <bool ROPE>
struct StGeo {
    static constexpr int kStage = (ROPE ? 3 : 2) * kStTile;
    static constexpr int kStages = kStRing / kStage;       // 4 or 6
};

constexpr int kApXWarps = 8;
constexpr int kApEWarps = 8;
constexpr int kApXThreads = 32 * kApXWarps;
constexpr int kApThreads = 32 * (3 + kApXWarps + kApEWarps);   // + the G producer warp
constexpr int kApORows = 32;                      // rows of o one epilogue warp stores
constexpr int kApTmemCols = 256;
// tc_apply_kernel modes: the gated apply, and for the backward the raw
// product, the gate terms and the masked gradient
constexpr int kApGate = 0, kApRaw = 1, kApTerms = 2, kApGrad = 3;
static_assert(kApGate == kApplyGate && kApRaw == kApplyRaw && kApTerms == kApplyTerms &&
                  kApGrad == kApplyGrad,
              "apply modes of the launcher");

// Ring geometry of the apply kernel per mode: Q stages, G stages, the bytes
// of a G stage and the den slots.  The gate terms stage g and dout tiles
// together, in two stages of each ring.  The masked gradient holds a Q tile
// only from its load to its MMA (two stages), and gives the third stage's
// room to the RoPE rows on their way to TMEM.  The raw product reads only Q:
// its G slots just stage the output, two of them suffice (a slot is refilled
// once the store of the tile before has read it), and the third becomes a
// fourth Q stage, so more of the one input stream is in flight.
template <int MODE>
struct ApGeo {
    static constexpr int kQS = MODE == kApTerms || MODE == kApGrad ? 2
                               : MODE == kApRaw                    ? kApQStages + 1
                                                                   : kApQStages;
    static constexpr int kGS = MODE == kApTerms || MODE == kApRaw ? 2 : kApGStages;
    static constexpr int kGT = MODE == kApTerms ? 2 * kApTile : kApTile;
    static constexpr int kDS = MODE == kApTerms ? 2 : kApDSlots;   // den slots
};
constexpr int kApRowsPerThread = kApTok * 16 / kApXThreads;   // 8

static_assert(kStRowsPerThread == 4 && kApRowsPerThread == 8, "thread/tile split");

// Units [start(c), start(c+1)) belong to CTA c.
struct Split {
    long long U;
    int G;
    __host__ __device__ long long start(int c) const { return (long long)c * U / G; }
    // The CTA whose range holds unit u.
    __host__ __device__ int owner(long long u) const {
        return (int)(((u + 1) * (long long)G - 1) / U);
    }
};

__device__ __forceinline__ uint32_t relu_bf2(uint32_t x) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&x);
    h = __hmax2(h, __floats2bfloat162_rn(0.f, 0.f));
    return *reinterpret_cast<uint32_t*>(&h);
}

// The eight bf16 values of a 16-byte chunk as floats (element 2p in the low half).
__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// The four (cos, sin) pairs of one 16-byte chunk, stored as fp16 pairs.
__device__ __forceinline__ void unpack_cs(const uint4& w, float2 (&cs)[4]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) cs[i] = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
}

// Rotates the pairs of f (phi of one chunk) and returns them packed as bf16.
__device__ __forceinline__ uint4 rotate_chunk(const float (&f)[8], const float2 (&cs)[4]) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = f[2 * i] * cs[i].x - f[2 * i + 1] * cs[i].y;
        const float b = f[2 * i] * cs[i].y + f[2 * i + 1] * cs[i].x;
        o[i] = f2_to_bf2(a, b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// A wait taken by all 32 lanes of a warp: the warp proceeds only if every
// lane saw the phase complete, so the lanes never split on an abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Eight outputs o = num / (den * (1 + exp(-g))) = sigmoid(g) * num / den of
// one 16-byte chunk of g, with den = phi(q) . z + eps of the row and num the
// eight fp32 numerators.  exp(-g) = 2^(-g log2 e); a gate far below zero
// gives exp(-g) = +inf and o = 0, far above zero exp(-g) = 0 and o = num / den.
__device__ __forceinline__ uint4 gate_chunk(uint4 g8, const uint32_t* num, float den) {
    constexpr float kLog2e = 1.4426950408889634f;
    const float2 dd = make_float2(den, den);
    const float2 kl = make_float2(-kLog2e, -kLog2e);
    const uint32_t w[4] = {g8.x, g8.y, g8.z, g8.w};
    uint32_t ow[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 gp = make_float2(__uint_as_float(w[e] << 16),
                                      __uint_as_float(w[e] & 0xffff0000u));
        const float2 t = mul2(gp, kl);
        const float2 d = fma2(dd, make_float2(ex2_approx(t.x), ex2_approx(t.y)), dd);
        const float2 o = mul2(make_float2(__uint_as_float(num[2 * e]),
                                          __uint_as_float(num[2 * e + 1])),
                              make_float2(rcp_approx(d.x), rcp_approx(d.y)));
        ow[e] = f2_to_bf2(o.x, o.y);
    }
    return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// The gate terms of eight elements of one row: g8 and d8 hold g and dout,
// num the eight fp32 numerators, inv_den 1 / den of the row.  With s =
// sigmoid(g) (as in gate_chunk): a = dout s / den (to a8), dg = dout num
// s (1 - s) / den (to g8o), and part += a . num.
__device__ __forceinline__ void terms_chunk(uint4 g8, uint4 d8, const uint32_t* num,
                                            float inv_den, uint4& a8, uint4& g8o, float& part) {
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
    const uint32_t dw[4] = {d8.x, d8.y, d8.z, d8.w};
    uint32_t aw[4], ow[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 gp = make_float2(__uint_as_float(gw[e] << 16),
                                      __uint_as_float(gw[e] & 0xffff0000u));
        const float2 dp = make_float2(__uint_as_float(dw[e] << 16),
                                      __uint_as_float(dw[e] & 0xffff0000u));
        const float2 np = make_float2(__uint_as_float(num[2 * e]), __uint_as_float(num[2 * e + 1]));
        const float2 t = mul2(gp, make_float2(-kLog2e, -kLog2e));
        const float2 e2 = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        const float2 sg = make_float2(rcp_approx(1.f + e2.x), rcp_approx(1.f + e2.y));
        const float2 av = mul2(mul2(dp, make_float2(inv_den, inv_den)), sg);   // a
        const float2 one_m = make_float2(1.f - sg.x, 1.f - sg.y);
        const float2 gv = mul2(mul2(av, np), one_m);                           // dg
        part = fmaf(av.x, np.x, fmaf(av.y, np.y, part));
        aw[e] = f2_to_bf2(av.x, av.y);
        ow[e] = f2_to_bf2(gv.x, gv.y);
    }
    a8 = make_uint4(aw[0], aw[1], aw[2], aw[3]);
    g8o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// Eight elements of a masked gradient row: out = [x > 0] (R^T y + w z), with
// x8 the bf16 input whose feature map is differentiated, y the eight fp32
// products of the tensor cores, cs4 the four (cos, sin) fp16 pairs of the
// chunk (R^T turns each pair back: (y0 c + y1 s, -y0 s + y1 c)) when ROPE,
// w the row's weight and z8 the eight matching entries of z.
template <bool ROPE>
__device__ __forceinline__ uint4 grad_chunk(uint4 x8, const uint32_t* y, uint4 cs4, float w,
                                            const float* z8) {
    float f[8];
    unpack8(x8, f);
    float yv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) yv[j] = __uint_as_float(y[j]);
    if (ROPE) {
        float2 cs[4];
        unpack_cs(cs4, cs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = yv[2 * i], b = yv[2 * i + 1];
            yv[2 * i] = a * cs[i].x + b * cs[i].y;
            yv[2 * i + 1] = b * cs[i].x - a * cs[i].y;
        }
    }
    const float4 za = *reinterpret_cast<const float4*>(z8);
    const float4 zb = *reinterpret_cast<const float4*>(z8 + 4);
    const float zv[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = f[2 * i] > 0.f ? fmaf(w, zv[2 * i], yv[2 * i]) : 0.f;
        const float b = f[2 * i + 1] > 0.f ? fmaf(w, zv[2 * i + 1], yv[2 * i + 1]) : 0.f;
        o[i] = f2_to_bf2(a, b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// warp_wait for phases completed by arrivals from other CTAs of the cluster.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, unsigned* status) {
    const bool ok = mbar_wait_cluster(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Offset of 16-byte chunk c (dims 8c..8c+7) of row r in a 128-byte-swizzled
// tile made of two 64-column boxes of `half` bytes each.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int c, int half) {
    return (uint32_t)((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Counts one contributor of a head for launch `epoch`; a count left by an
// earlier launch (another epoch) counts as zero.  Returns the new count, or 0
// if the atomic kept failing (status raised).  A launch that completes leaves
// every counter it used at zero (see the flush warps), so the tag matters only
// after a launch that gave up a wait.
__device__ inline uint32_t count_contributor(unsigned long long* ctr, uint32_t epoch, unsigned* status) {
    unsigned long long seen = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (int it = 0; it < (1 << 20); ++it) {
        const unsigned long long want = (uint32_t)(seen >> 32) == epoch
                                            ? seen + 1ull
                                            : (((unsigned long long)epoch << 32) | 1ull);
        const unsigned long long got = atomicCAS(ctr, seen, want);
        if (got == seen) return (uint32_t)want;
        seen = got;
    }
    raise_status(status, kStatusTimeout);
    return 0;
}

// Waits until the head's counter shows k contributors for launch `epoch`.
// Every contributor is resident (the state kernel is a cooperative launch) and
// counts itself without waiting for anyone, so the wait ends; it still gives
// up after kWaitLimitNs.
__device__ inline bool wait_count(const unsigned long long* ctr, uint32_t epoch, uint32_t k,
                           volatile int* abort, unsigned* status) {
    const uint64_t t0 = global_ns();
    for (;;) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if ((uint32_t)(v >> 32) == epoch && (uint32_t)v >= k) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            raise_status(status, kStatusTimeout);
            *abort = 1;
            return false;
        }
        __nanosleep(100);
    }
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// A [BH][N][128] bf16 tensor seen as 3D (d fastest), boxes of 64 columns x
// `rows` tokens x 1 head, 128-byte swizzle; rows past N read as zero and are
// not written by stores.
inline bool make_map(CUtensorMap* m, const void* base, int N, int BH, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)N * kRowBytes};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The per-token RoPE rows, [N][64] 4-byte (cos, sin) fp16 pairs, 256 bytes per
// token, boxes of `rows` tokens; rows past N read as zero.
inline bool make_rope_map(CUtensorMap* m, const uint32_t* base, int N, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kPairs, (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)kPairs * 4};
    cuuint32_t box[2] = {(cuuint32_t)kPairs, (cuuint32_t)rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The per-token RoPE rows again, in boxes of 32 words (128 bytes: half a
// token's pairs) x 32 tokens with 128-byte swizzle: chunk c of box row r lands
// at r * 128 + ((c ^ (r & 7)) << 4).  Rows past N read as zero.
inline bool make_rope_box_map(CUtensorMap* m, const uint32_t* base, int N) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kPairs, (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)kPairs * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A tag for one launch of a kernel that counts contributors: distinct for
// every call (a count left by an earlier launch that gave up reads as zero).
uint32_t next_epoch();

}  // namespace tc
}  // namespace sla
