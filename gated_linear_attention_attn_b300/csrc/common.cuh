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

// Layout of a RoPE table buffer, in 4-byte words: the separable fp32
// (cos, sin) pairs of each axis ([T][dt/2], [Hs][dh/2], [Ws][dw/2]), then,
// from the next 256-byte boundary, one row per token of d/2 (cos, sin) pairs
// as two fp16 values in a word (cos in the low half).
inline size_t rope_sep_words(int T, int Hs, int Ws, int dt, int dh, int dw) {
    return (size_t)T * dt + (size_t)Hs * dh + (size_t)Ws * dw;
}
inline size_t rope_tok_offset_words(int T, int Hs, int Ws, int dt, int dh, int dw) {
    return (rope_sep_words(T, Hs, Ws, dt, dh, dw) + 63) & ~size_t(63);
}
inline size_t rope_total_words(int T, int Hs, int Ws, int dt, int dh, int dw) {
    return rope_tok_offset_words(T, Hs, Ws, dt, dh, dw) +
           (size_t)T * Hs * Ws * (size_t)((dt + dh + dw) / 2);
}

// Device view of a filled RoPE table: (cos, sin) pairs per axis, each axis
// [extent][band pairs], axes in the order t, h, w; and the per-token rows.
struct RopeView {
    const float2* tab_t;   // [T][pt]
    const float2* tab_h;   // [Hs][ph]
    const float2* tab_w;   // [Ws][pw]
    const uint32_t* tok;   // [N][64] fp16 (cos, sin) per pair, 256 bytes per token
    int T, Hs, Ws;
    int pt, ph, pw;        // pairs per band: dt/2, dh/2, dw/2
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
