// Shared device helpers of the linear-attention library: the RoPE table view,
// the device status word, bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sla {

constexpr int kHeadDim = 128;          // d: 128 in both the 5B and the 14B models
constexpr int kPairs = kHeadDim / 2;

// Bits of the device status word (one 32-bit word per device).
constexpr unsigned kStatusTimeout = 1u;   // a bounded wait gave up
constexpr unsigned kStatusLayout = 2u;    // shared memory not 1 KB aligned: nothing ran

// Division of 0 <= n < 2^31 by an invariant divisor d >= 1 with one high
// multiply, after Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, floor(n / d) = (umulhi(n, m) + n) >> s.
// The sum cannot overflow because umulhi(n, m) < n < 2^31.
struct FastDiv {
    uint32_t mul = 1;
    uint32_t shift = 0;
};

inline FastDiv make_fastdiv(int d) {
    FastDiv f;
    uint32_t s = 0;
    while ((1ull << s) < (unsigned long long)d) ++s;
    const unsigned long long pow2 = 1ull << s;
    f.mul = (uint32_t)(((1ull << 32) * (pow2 - (unsigned long long)d)) / (unsigned long long)d + 1);
    f.shift = s;
    return f;
}

__device__ __forceinline__ int fast_div(int n, FastDiv f) {
    return (int)((__umulhi((uint32_t)n, f.mul) + (uint32_t)n) >> f.shift);
}

// Device view of a filled RoPE table: (cos, sin) pairs per axis, each axis
// [extent][band pairs], axes in the order t, h, w.
struct RopeView {
    const float2* tab_t;   // [T][pt]
    const float2* tab_h;   // [Hs][ph]
    const float2* tab_w;   // [Ws][pw]
    int T, Hs, Ws;
    int pt, ph, pw;        // pairs per band: dt/2, dh/2, dw/2
    FastDiv div_ws, div_hs;   // n / Ws and (n / Ws) / Hs
};

// Grid coordinates of token n: n = (t*Hs + h)*Ws + w.
struct TokenPos {
    int t, h, w;
};

__device__ __forceinline__ TokenPos token_pos(const RopeView& r, int n) {
    TokenPos p;
    int hw = n / r.Ws;
    p.w = n - hw * r.Ws;
    p.t = hw / r.Hs;
    p.h = hw - p.t * r.Hs;
    return p;
}

// (cos, sin) of pair p (0 <= p < 64) for a token at `pos`.
__device__ __forceinline__ float2 rope_cs(const RopeView& r, const TokenPos& pos, int p) {
    if (p < r.pt) return __ldg(r.tab_t + (size_t)pos.t * r.pt + p);
    p -= r.pt;
    if (p < r.ph) return __ldg(r.tab_h + (size_t)pos.h * r.ph + p);
    p -= r.ph;
    return __ldg(r.tab_w + (size_t)pos.w * r.pw + p);
}

// Complex rotation of the pair (x0, x1) by (c, s).
__device__ __forceinline__ void rotate_pair(float& x0, float& x1, float2 cs) {
    float a = x0 * cs.x - x1 * cs.y;
    float b = x0 * cs.y + x1 * cs.x;
    x0 = a;
    x1 = b;
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
}

__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void raise_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Any wait inside a kernel gives up after this many nanoseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

}  // namespace sla
