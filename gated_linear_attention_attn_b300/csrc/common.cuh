// Shared device helpers of the linear-attention library: the RoPE table
// layout and view, the device status word, bf16 packing.
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
constexpr unsigned kStatusBadTable = 4u;  // a RoPE table's header does not fit the call

// Layout of a RoPE table buffer, in 4-byte words, for a grid of N tokens and
// head dimension d (P = d/2 pairs):
//   [0, 64)                 header (kRopeHdr* below)
//   [64, 64 + N*P)          per-token rows: pair p of token n is one word,
//                           fp16 cos in the low half, fp16 sin in the high half
//   [64 + N*P, 64 + 3*N*P)  per-token pairs [N][P][2] as fp32 (cos, sin)
constexpr int kRopeHeaderWords = 64;
constexpr uint32_t kRopeMagic = 0x33414c53u;     // "SLA3" in little-endian bytes
constexpr uint32_t kRopeVersion = 1u;
// header words
constexpr int kRopeHdrMagic = 0, kRopeHdrVersion = 1, kRopeHdrN = 2, kRopeHdrD = 3;
constexpr int kRopeHdrT = 4, kRopeHdrHs = 5, kRopeHdrWs = 6;
constexpr int kRopeHdrDt = 7, kRopeHdrDh = 8, kRopeHdrDw = 9, kRopeHdrBase = 10;
constexpr int kRopeHdrRows = 11, kRopeHdrPairs = 12;   // word offsets of the two parts

inline size_t rope_total_words(long long N, int d) {
    return (size_t)kRopeHeaderWords + (size_t)N * (size_t)(d / 2) * 3;
}

// Device view of a RoPE table: which tokens a launch reads and which head
// dimension it expects.  The kernels check the header against it before they
// read anything else of the table (rope_table_ok).
struct RopeView {
    const uint32_t* hdr;   // the table: header, fp16 rows, fp32 pairs
    const uint32_t* tok;   // the fp16 rows (hdr + kRopeHeaderWords): [tokens][d/2]
    int need;              // the launch reads tokens [0, need) of the table
    int exact;             // nonzero: the table must have exactly `need` tokens
    int d;                 // head dimension the table must be built for
};

// The header written by sla_rope_table_fill / sla_rope_table_from_pairs, and
// enough tokens for the launch.
__device__ __forceinline__ bool rope_table_ok(const RopeView& r) {
    if (!r.hdr) return false;
    const uint32_t magic = __ldg(r.hdr + kRopeHdrMagic);
    const uint32_t ver = __ldg(r.hdr + kRopeHdrVersion);
    const uint32_t n = __ldg(r.hdr + kRopeHdrN);
    const uint32_t d = __ldg(r.hdr + kRopeHdrD);
    const uint32_t rows = __ldg(r.hdr + kRopeHdrRows);
    const uint32_t pairs = __ldg(r.hdr + kRopeHdrPairs);
    if (magic != kRopeMagic || ver != kRopeVersion || d != (uint32_t)r.d) return false;
    if (rows != (uint32_t)kRopeHeaderWords || pairs != rows + n * (d / 2)) return false;
    return r.exact ? n == (uint32_t)r.need : n >= (uint32_t)r.need;
}

// The fp32 (cos, sin) pairs of the table, [tokens][d/2].
__device__ __forceinline__ const float2* rope_pairs(const RopeView& r) {
    return reinterpret_cast<const float2*>(r.hdr + __ldg(r.hdr + kRopeHdrPairs));
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
