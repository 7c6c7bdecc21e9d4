// bf16 path of the linear-attention forward on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Two persistent launches, each splitting its work units evenly over at most
// one CTA per SM ("stream-K": a CTA's range of units may cross a head):
//
//   tc_state_kernel   units = (head, 64-token tile).  Warp 0 streams K and V
//                     tiles into a 6-stage ring; eight transform warps apply
//                     phi = ReLU (and the 3D RoPE) to the K tile in shared
//                     memory, in place, and sum z = sum phi(k) (unrotated) in
//                     registers; one thread of warp 1 issues
//                     S^T += (phi~(K)^T V)^T on the tensor core (M = N = 128,
//                     K = 64 tokens, both operands MN-major).  When a CTA
//                     leaves a head it writes its partial (S^T, z) in fp32 to
//                     workspace slot (cta + head) and counts itself in the
//                     head's counter; the last contributor of a head sums the
//                     head's slots in a fixed order and writes the head's
//                     state: S^T in bf16, already in the tensor-core layout of
//                     the apply kernel's B operand, and z in fp32.
//   tc_apply_kernel   units = (head, 128-token tile).  Warp 0 streams Q and G
//                     tiles into a 3-stage ring and, once per head, the head's
//                     state with one bulk copy.  Eight transform warps apply
//                     phi and RoPE to the Q tile in place and form
//                     den = phi(q) . z + eps; one thread of warp 1 issues
//                     num = phi~(Q) S (M = N = K = 128) into one of two TMEM
//                     accumulators; eight epilogue warps read num from TMEM,
//                     compute sigmoid(g) * num / den over the G tile in place,
//                     and one of them stores the tile with TMA.
//
// The apply kernel is launched as a programmatic dependent of the state
// kernel: it prefetches Q and G (which the state kernel does not write) and
// waits for the state kernel's completion only before its first state load.
//
// Every mbarrier wait gives up after about a second (status word + early
// return), and every exit path waits for the copies and MMAs it issued.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

using namespace ptx;

constexpr int kRowBytes = kHeadDim * 2;                          // one bf16 token row: 256 B
// A partial slot: S^T [128][128] fp32, then z as one 128-float part per
// transform warp of the state kernel.
constexpr int kStXWarps = 8;                                     // transform warps
constexpr int kPartialFloats = kHeadDim * kHeadDim + kStXWarps * kHeadDim;
constexpr int kStateSBytes = kHeadDim * kHeadDim * 2;            // S^T bf16: 32 KB
constexpr int kStateBytes = kStateSBytes + kHeadDim * 4;         // + z fp32: 33280 B
constexpr int kStateHalf = kStateSBytes / 2;                     // one 64-column half

// ---- state kernel geometry
constexpr int kStTok = 64;                        // tokens per tile
constexpr int kStStages = 6;
constexpr int kStHalf = kStTok * 128;             // one 64-column box: 8 KB
constexpr int kStTile = 2 * kStHalf;              // one tensor tile: 16 KB
constexpr int kStStage = 2 * kStTile;             // K + V: 32 KB
constexpr int kStXThreads = 32 * kStXWarps;
constexpr int kStThreads = 64 + kStXThreads;      // TMA warp, MMA warp, transform warps
constexpr int kStTmemCols = 256;                  // two 128-column accumulators
constexpr int kStRowsPerThread = kStTok * 16 / kStXThreads;   // 4

// ---- apply kernel geometry
constexpr int kApTok = 128;
constexpr int kApStages = 3;
constexpr int kApHalf = kApTok * 128;             // 16 KB
constexpr int kApTile = 2 * kApHalf;              // 32 KB
constexpr int kApStage = 2 * kApTile;             // Q + G: 64 KB
constexpr int kApXWarps = 8;
constexpr int kApEWarps = 8;
constexpr int kApXThreads = 32 * kApXWarps;
constexpr int kApThreads = 64 + 32 * (kApXWarps + kApEWarps);
constexpr int kApTmemCols = 256;
constexpr int kApRowsPerThread = kApTok * 16 / kApXThreads;   // 8
constexpr int kApFirstEpilogue = 64 + kApXThreads;            // thread index of the storer

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

struct StateParams {
    int N, Tk;                      // tokens per head, 64-token tiles per head
    Split split;
    RopeView rope;
    float* partial;                 // slot (cta + head), kPartialFloats each
    unsigned long long* counters;   // per head: (epoch << 32) | contributors counted
    uint8_t* state;                 // per head: kStateBytes
    uint32_t epoch;                 // distinct for every launch
    unsigned* status;
};

struct ApplyParams {
    int N, Tq;
    Split split;
    RopeView rope;
    const uint8_t* state;
    float eps;
    unsigned* status;
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

// Grid coordinates of token n: n = (t*Hs + h)*Ws + w.
__device__ __forceinline__ void grid_pos(const RopeView& r, int n, int& t, int& h, int& w) {
    const int hw = fast_div(n, r.div_ws);
    w = n - hw * r.Ws;
    t = fast_div(hw, r.div_hs);
    h = hw - t * r.Hs;
}

// RoPE of the four pairs of one 16-byte chunk (dims 8c..8c+7).  Pair p's
// (cos, sin) sits in the table of its band at the row given by the token's
// coordinate on that band's axis; the band of each pair is fixed per chunk,
// so it is resolved once and the per-token lookup has no branches.
struct ChunkRope {
    const float2* base[4];   // band table + pair index inside the band
    int stride[4];           // pairs per row of that band
    int axis[4];             // 0 = t, 1 = h, 2 = w

    __device__ __forceinline__ void init(const RopeView& r, int c) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = 4 * c + i;
            if (p < r.pt) {
                axis[i] = 0;
                base[i] = r.tab_t + p;
                stride[i] = r.pt;
            } else if (p < r.pt + r.ph) {
                axis[i] = 1;
                base[i] = r.tab_h + (p - r.pt);
                stride[i] = r.ph;
            } else {
                axis[i] = 2;
                base[i] = r.tab_w + (p - r.pt - r.ph);
                stride[i] = r.pw;
            }
        }
    }

    // Rotates the pairs of f (phi of one chunk) for the token at (t, h, w)
    // and returns them packed as bf16.
    __device__ __forceinline__ uint4 rotate(const float (&f)[8], int t, int h, int w) const {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int coord = axis[i] == 0 ? t : (axis[i] == 1 ? h : w);
            const float2 cs = __ldg(base[i] + coord * stride[i]);
            const float a = f[2 * i] * cs.x - f[2 * i + 1] * cs.y;
            const float b = f[2 * i] * cs.y + f[2 * i + 1] * cs.x;
            o[i] = f2_to_bf2(a, b);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

// A wait taken by all 32 lanes of a warp: the warp proceeds only if every
// lane saw the phase complete, so the lanes never split on an abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Offset of 16-byte chunk c (dims 8c..8c+7) of row r in a 128-byte-swizzled
// tile made of two 64-column boxes of `half` bytes each.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int c, int half) {
    return (uint32_t)((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Counts one contributor of a head for launch `epoch`; a count left by an
// earlier launch (another epoch) counts as zero.  Returns the new count, or 0
// if the atomic kept failing (status raised).
__device__ uint32_t count_contributor(unsigned long long* ctr, uint32_t epoch, unsigned* status) {
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

// =================================================================== state ==

template <bool ROPE>
__global__ void __launch_bounds__(kStThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                StateParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStStages * kStStage);
    uint64_t* kready = full + kStStages;
    uint64_t* empty = kready + kStStages;
    uint64_t* accfull = empty + kStStages;        // [2]
    uint64_t* accempty = accfull + 2;             // [2]
    uint64_t* slotdone = accempty + 2;            // a segment's slot is written
    uint64_t* lastknown = slotdone + 1;           // the head's last contributor is known
    uint64_t* mma_done = lastknown + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = p.split.start(cta), u1 = p.split.start(cta + 1);
    const uint32_t smem0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&kready[s], kStXWarps);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], kStXWarps);
        }
        mbar_init(slotdone, kStXWarps);
        mbar_init(lastknown, 1);
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;    // the swizzled tiles need 1 KB alignment
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        griddep_launch_dependents();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kStTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            long long it = 0;
            for (long long u = u0; u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tk), tile = (int)(u % p.Tk);
                const int s = (int)(it % kStStages);
                const uint32_t round = (uint32_t)(it / kStStages);
                if (!mbar_wait(&empty[s], (round & 1) ^ 1, abort_flag, p.status)) break;
                uint8_t* st = smem + s * kStStage;
                mbar_arrive_expect_tx(&full[s], kStStage);
                tma_load_3d(st, &tm_k, &full[s], 0, tile * kStTok, h, policy);
                tma_load_3d(st + kStHalf, &tm_k, &full[s], 64, tile * kStTok, h, policy);
                tma_load_3d(st + kStTile, &tm_v, &full[s], 0, tile * kStTok, h, policy);
                tma_load_3d(st + kStTile + kStHalf, &tm_v, &full[s], 64, tile * kStTok, h,
                            policy);
            }
            // every load issued has landed before the CTA may exit
            const long long first = it > kStStages ? it - kStStages : 0;
            for (long long j = first; j < it; ++j)
                mbar_wait_drain(&full[j % kStStages], (uint32_t)((j / kStStages) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, true, true);
            long long it = 0;
            int seg = -1, cur_h = -1;
            bool ok = !*abort_flag, first = false;
            for (long long u = u0; ok && u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tk);
                const int s = (int)(it % kStStages);
                const uint32_t round = (uint32_t)(it / kStStages);
                if (h != cur_h) {
                    if (seg >= 0) mma_commit(&accfull[seg & 1]);
                    ++seg;
                    cur_h = h;
                    first = true;
                    ok = mbar_wait(&accempty[seg & 1], ((seg >> 1) & 1) ^ 1, abort_flag,
                                   p.status);
                    if (!ok) break;
                }
                ok = mbar_wait(&kready[s], round & 1, abort_flag, p.status) &&
                     mbar_wait(&full[s], round & 1, abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kb = smem0 + s * kStStage, vb = kb + kStTile;
#pragma unroll
                for (int ks = 0; ks < kStTok / 16; ++ks) {
                    // 16 tokens = two 8-row swizzle atoms; the two 64-wide halves
                    // of M (and N) sit kStHalf apart
                    const uint64_t a = smem_desc_sw128(kb + ks * 2048, kStHalf, 1024);
                    const uint64_t b = smem_desc_sw128(vb + ks * 2048, kStHalf, 1024);
                    mma_bf16(tmem + (uint32_t)(seg & 1) * 128, a, b, idesc,
                             (first && ks == 0) ? 0u : 1u);
                }
                first = false;
                mma_commit(&empty[s]);
            }
            if (ok && seg >= 0) mma_commit(&accfull[seg & 1]);
            // nothing of ours is in flight once this barrier fires
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0);
        }
    } else {
        // ------------------------------------------------ transform + flush + merge
        const int tt = threadIdx.x - 64;           // 0..255
        const int c = tt & 15, rl = tt >> 4;        // chunk (dims 8c..8c+7), row lane 0..15
        const int xw = warp - 2;                    // transform warp 0..7
        float zacc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
        ChunkRope cr;
        if (ROPE) cr.init(p.rope, c);
        long long it = 0;
        int seg = -1, cur_h = -1;
        bool ok = !*abort_flag;

        // The head's state from its partial slots, summed in slot order.
        auto merge = [&](int hh) {
            const int lo = p.split.owner((long long)hh * p.Tk);
            const int hi = p.split.owner((long long)(hh + 1) * p.Tk - 1);
            uint8_t* dst = p.state + (size_t)hh * kStateBytes;
            float4 acc[8][2];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[i][0] = acc[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cc = lo; cc <= hi; ++cc) {
                const float* src = p.partial + (size_t)(cc + hh) * kPartialFloats + c * 8;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + (rl + 16 * i) * 128);
                    const float4 a = __ldcg(s4), b = __ldcg(s4 + 1);
                    acc[i][0].x += a.x; acc[i][0].y += a.y; acc[i][0].z += a.z; acc[i][0].w += a.w;
                    acc[i][1].x += b.x; acc[i][1].y += b.y; acc[i][1].z += b.z; acc[i][1].w += b.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int n = rl + 16 * i;
                uint4 w;
                w.x = f2_to_bf2(acc[i][0].x, acc[i][0].y);
                w.y = f2_to_bf2(acc[i][0].z, acc[i][0].w);
                w.z = f2_to_bf2(acc[i][1].x, acc[i][1].y);
                w.w = f2_to_bf2(acc[i][1].z, acc[i][1].w);
                *reinterpret_cast<uint4*>(dst + sw128_off(n, c, kStateHalf)) = w;
            }
            if (tt < kHeadDim) {
                float zs = 0.f;
                for (int cc = lo; cc <= hi; ++cc) {
                    const float* zp = p.partial + (size_t)(cc + hh) * kPartialFloats +
                                      kHeadDim * kHeadDim + tt;
#pragma unroll
                    for (int w8 = 0; w8 < kStXWarps; ++w8) zs += __ldcg(zp + w8 * kHeadDim);
                }
                reinterpret_cast<float*>(dst + kStateSBytes)[tt] = zs;
            }
        };

        // S^T and z of this CTA's share of head hh -> slot (cta + hh); the
        // head's last contributor then merges.  The warps meet only on
        // mbarriers with bounded waits, so a warp that gives up cannot strand
        // the others.
        auto flush = [&](int sg, int hh) -> bool {
            const bool got = warp_wait(&accfull[sg & 1], (sg >> 1) & 1, abort_flag, p.status);
            float* slot = p.partial + (size_t)(cta + hh) * kPartialFloats;
            if (got) {
                tc_fence_after();
                const int quad = warp & 3, hf = xw >> 2;   // TMEM lanes 32*quad.., columns 64*hf..
                const int m = 32 * quad + lane;
#pragma unroll 1
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(sg & 1) * 128 +
                                  hf * 64 + ch * 32,
                              r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        slot[(size_t)(hf * 64 + ch * 32 + j) * kHeadDim + m] =
                            __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[sg & 1]);
            }
            // this warp's z: lanes l and l^16 hold the same dims for neighbouring rows
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 16);
            if (lane < 16) {
                float4* zp = reinterpret_cast<float4*>(slot + kHeadDim * kHeadDim +
                                                       xw * kHeadDim + c * 8);
                zp[0] = make_float4(zacc[0], zacc[1], zacc[2], zacc[3]);
                zp[1] = make_float4(zacc[4], zacc[5], zacc[6], zacc[7]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
            __threadfence();
            __syncwarp();
            if (!got) return false;
            if (lane == 0) mbar_arrive(slotdone);
            if (tt == 0) {
                // every warp's share of the slot is written: count this CTA in
                const bool done = mbar_wait(slotdone, sg & 1, abort_flag, p.status);
                int last = 0;
                if (done) {
                    __threadfence();
                    const int lo = p.split.owner((long long)hh * p.Tk);
                    const int hi = p.split.owner((long long)(hh + 1) * p.Tk - 1);
                    const uint32_t n = count_contributor(p.counters + hh, p.epoch, p.status);
                    last = n == (uint32_t)(hi - lo + 1) ? 1 : 0;
                    __threadfence();
                }
                *last_flag = last;
                mbar_arrive(lastknown);
            }
            if (!warp_wait(lastknown, sg & 1, abort_flag, p.status)) return false;
            if (*last_flag) {
                __threadfence();
                merge(hh);
            }
            return true;
        };

        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tk), tile = (int)(u % p.Tk);
            if (h != cur_h) {
                if (seg >= 0 && !(ok = flush(seg, cur_h))) break;
                ++seg;
                cur_h = h;
            }
            const int s = (int)(it % kStStages);
            const uint32_t round = (uint32_t)(it / kStStages);
            if (!(ok = warp_wait(&full[s], round & 1, abort_flag, p.status))) break;
            const uint32_t kb = smem0 + s * kStStage;
            const int n0 = tile * kStTok;
#pragma unroll
            for (int i = 0; i < kStRowsPerThread; ++i) {
                const int r = rl + 16 * i;
                const uint32_t addr = kb + sw128_off(r, c, kStHalf);
                uint4 x = lds128(addr);
                x.x = relu_bf2(x.x);
                x.y = relu_bf2(x.y);
                x.z = relu_bf2(x.z);
                x.w = relu_bf2(x.w);
                float f[8];
                unpack8(x, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) zacc[j] += f[j];
                if (ROPE) {
                    // rows past N are zero (TMA fill): any in-range position will do
                    int t, hh, w;
                    grid_pos(p.rope, min(n0 + r, p.N - 1), t, hh, w);
                    x = cr.rotate(f, t, hh, w);
                }
                sts128(addr, x);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&kready[s]);
        }
        if (ok && seg >= 0) flush(seg, cur_h);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kStTmemCols);
    }
}

// =================================================================== apply ==

template <bool ROPE>
__global__ void __launch_bounds__(kApThreads, 1)
tc_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o, ApplyParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sbuf = smem + kApStages * kApStage;               // S^T bf16 (B operand), then z
    float* zs = reinterpret_cast<float*>(sbuf + kStateSBytes);  // [128]
    float* dens = zs + kHeadDim;                                // [stages][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(dens + kApStages * kApTok);
    uint64_t* qready = full + kApStages;
    uint64_t* empty = qready + kApStages;
    uint64_t* ogather = empty + kApStages;
    uint64_t* accfull = ogather + kApStages;    // [2]
    uint64_t* accempty = accfull + 2;           // [2]
    uint64_t* sready = accempty + 2;
    uint64_t* sfree = sready + 1;
    uint64_t* mma_done = sfree + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = p.split.start(cta), u1 = p.split.start(cta + 1);
    const uint32_t smem0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kApStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&qready[s], kApXWarps);
            mbar_init(&empty[s], 1);
            mbar_init(&ogather[s], kApEWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], kApEWarps);
        }
        mbar_init(sready, 1);
        mbar_init(sfree, 1 + kApXWarps);
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_o);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kApTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            // The first head's state is written by the preceding launch: its load
            // waits for that launch to complete, after the first Q/G tiles are in
            // flight.  Later heads wait until the previous state is no longer read.
            int first_h = -1, loads = 0;
            bool first_pending = true;
            auto load_state = [&](int hh) {
                ++loads;
                mbar_arrive_expect_tx(sready, kStateBytes);
                bulk_load(sbuf, p.state + (size_t)hh * kStateBytes, kStateBytes, sready);
            };
            auto load_first = [&]() {
                griddep_wait();
                load_state(first_h);
                first_pending = false;
            };
            long long it = 0;
            int heads = 0, cur_h = -1;
            bool ok = true;
            for (long long u = u0; u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
                if (h != cur_h) {
                    if (heads == 0) {
                        first_h = h;
                    } else {
                        if (first_pending) load_first();
                        if (!(ok = mbar_wait(sfree, (heads - 1) & 1, abort_flag, p.status)))
                            break;
                        load_state(h);
                    }
                    ++heads;
                    cur_h = h;
                }
                if (first_pending && it == kApStages) load_first();
                const int s = (int)(it % kApStages);
                const uint32_t round = (uint32_t)(it / kApStages);
                if (!(ok = mbar_wait(&empty[s], (round & 1) ^ 1, abort_flag, p.status))) break;
                uint8_t* st = smem + s * kApStage;
                mbar_arrive_expect_tx(&full[s], kApStage);
                tma_load_3d(st, &tm_q, &full[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_q, &full[s], 64, tile * kApTok, h, policy);
                tma_load_3d(st + kApTile, &tm_g, &full[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApTile + kApHalf, &tm_g, &full[s], 64, tile * kApTok, h,
                            policy);
            }
            if (ok && first_pending && first_h >= 0) load_first();
            // every copy issued has landed before the CTA may exit
            const long long first = it > kApStages ? it - kApStages : 0;
            for (long long j = first; j < it; ++j)
                mbar_wait_drain(&full[j % kApStages], (uint32_t)((j / kApStages) & 1));
            if (loads > 0) mbar_wait_drain(sready, (loads - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
            const uint32_t sb = smem_u32(sbuf);
            long long it = 0;
            int heads = 0, cur_h = -1;
            bool ok = !*abort_flag;
            for (long long u = u0; ok && u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tq);
                if (h != cur_h) {
                    if (heads > 0) mma_commit(sfree);      // old state no longer read
                    ok = mbar_wait(sready, heads & 1, abort_flag, p.status);
                    if (!ok) break;
                    ++heads;
                    cur_h = h;
                }
                const int s = (int)(it % kApStages);
                const uint32_t round = (uint32_t)(it / kApStages);
                const int a = (int)(it & 1);
                const uint32_t around = (uint32_t)(it >> 1);
                ok = mbar_wait(&accempty[a], (around & 1) ^ 1, abort_flag, p.status) &&
                     mbar_wait(&qready[s], round & 1, abort_flag, p.status) &&
                     mbar_wait(&full[s], round & 1, abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qb = smem0 + s * kApStage;
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                    // K-major, 128-byte swizzle: 16 k-values = 32 bytes inside a row
                    const uint32_t off = (ks >> 2) * kApHalf + (ks & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(qb + off, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(sb + off, 16, 1024);
                    mma_bf16(tmem + (uint32_t)a * 128, ad, bd, idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(&accfull[a]);
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0);
        }
    } else if (warp < 2 + kApXWarps) {
        // ------------------------------------------------ transform: phi, RoPE, den
        const int tt = threadIdx.x - 64;            // 0..255
        const int c = tt & 15, rl = tt >> 4;         // chunk, row lane 0..15
        ChunkRope cr;
        if (ROPE) cr.init(p.rope, c);
        float zc[8];
        long long it = 0;
        int heads = 0, cur_h = -1;
        bool ok = !*abort_flag;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
            if (h != cur_h) {
                if (!(ok = warp_wait(sready, heads & 1, abort_flag, p.status))) break;
                const float4 za = *reinterpret_cast<const float4*>(zs + 8 * c);
                const float4 zb = *reinterpret_cast<const float4*>(zs + 8 * c + 4);
                zc[0] = za.x; zc[1] = za.y; zc[2] = za.z; zc[3] = za.w;
                zc[4] = zb.x; zc[5] = zb.y; zc[6] = zb.z; zc[7] = zb.w;
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree);       // z of this head is in registers
                ++heads;
                cur_h = h;
            }
            const int s = (int)(it % kApStages);
            const uint32_t round = (uint32_t)(it / kApStages);
            if (!(ok = warp_wait(&full[s], round & 1, abort_flag, p.status))) break;
            const uint32_t qb = smem0 + s * kApStage;
            const int n0 = tile * kApTok;
            float den[kApRowsPerThread];
#pragma unroll
            for (int i = 0; i < kApRowsPerThread; ++i) {
                const int r = rl + 16 * i;
                const uint32_t addr = qb + sw128_off(r, c, kApHalf);
                uint4 x = lds128(addr);
                x.x = relu_bf2(x.x);
                x.y = relu_bf2(x.y);
                x.z = relu_bf2(x.z);
                x.w = relu_bf2(x.w);
                float f[8];
                unpack8(x, f);
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) d = fmaf(f[j], zc[j], d);
                den[i] = d;
                if (ROPE) {
                    int t, hh, w;
                    grid_pos(p.rope, min(n0 + r, p.N - 1), t, hh, w);
                    x = cr.rotate(f, t, hh, w);
                }
                sts128(addr, x);
            }
            // Sum den over the 16 chunk lanes of each row: each step halves the
            // rows a lane holds, so lane c ends with row rl + 16*(c >> 1).
            {
                const bool b3 = (c >> 3) & 1, b2 = (c >> 2) & 1, b1 = (c >> 1) & 1;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float send = b3 ? den[k] : den[k + 4];
                    const float keep = b3 ? den[k + 4] : den[k];
                    den[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float send = b2 ? den[k] : den[k + 2];
                    const float keep = b2 ? den[k + 2] : den[k];
                    den[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                {
                    const float send = b1 ? den[0] : den[1];
                    const float keep = b1 ? den[1] : den[0];
                    den[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
                den[0] += __shfl_xor_sync(0xffffffffu, den[0], 1);
                if ((c & 1) == 0) dens[s * kApTok + rl + 16 * (c >> 1)] = den[0] + p.eps;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&qready[s]);
        }
    } else {
        // ------------------------------------------------ epilogue: gate, divide, store
        const int ew = warp - 2 - kApXWarps;        // 0..7
        const int quad = warp & 3, hf = ew >> 2;     // TMEM lanes 32*quad.., columns 64*hf..
        const int r = 32 * quad + lane;              // TMEM lane = token row of the tile
        const bool storer = threadIdx.x == kApFirstEpilogue;
        long long it = 0;
        bool ok = !*abort_flag;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
            const int s = (int)(it % kApStages);
            const uint32_t round = (uint32_t)(it / kApStages);
            const int a = (int)(it & 1);
            const uint32_t around = (uint32_t)(it >> 1);
            ok = warp_wait(&accfull[a], around & 1, abort_flag, p.status) &&
                 warp_wait(&qready[s], round & 1, abort_flag, p.status) &&
                 warp_wait(&full[s], round & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const float rden = 1.f / dens[s * kApTok + r];
            const uint32_t gb = smem0 + s * kApStage + kApTile;
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)a * 128 + hf * 64 +
                              ch * 32,
                          v);
                tmem_ld_wait();
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    const uint32_t addr = gb + sw128_off(r, hf * 8 + ch * 4 + sub, kApHalf);
                    const uint4 gv = lds128(addr);
                    float gf[8];
                    unpack8(gv, gf);
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float o0 = __fdividef(__uint_as_float(v[sub * 8 + 2 * e]) * rden,
                                                    1.f + __expf(-gf[2 * e]));
                        const float o1 = __fdividef(__uint_as_float(v[sub * 8 + 2 * e + 1]) * rden,
                                                    1.f + __expf(-gf[2 * e + 1]));
                        ow[e] = f2_to_bf2(o0, o1);
                    }
                    sts128(addr, make_uint4(ow[0], ow[1], ow[2], ow[3]));
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&accempty[a]);
                mbar_arrive(&ogather[s]);
            }
            bool stored = true;
            if (storer) {
                stored = mbar_wait(&ogather[s], round & 1, abort_flag, p.status);
                if (stored) {
                    const uint8_t* ot = smem + s * kApStage + kApTile;
                    tma_store_3d(&tm_o, ot, 0, tile * kApTok, h);
                    tma_store_3d(&tm_o, ot + kApHalf, 64, tile * kApTok, h);
                    bulk_commit();
                    bulk_wait_read_all();          // the stage may be refilled after this
                    mbar_arrive(&empty[s]);
                }
            }
            if (!(ok = __all_sync(0xffffffffu, stored))) break;
        }
        if (storer) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kApTmemCols);
    }
}

// ==================================================================== host ==

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
bool make_map(CUtensorMap* m, const void* base, int N, int BH, int rows) {
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

constexpr size_t kStSmem = (size_t)kStStages * kStStage + 256;
constexpr size_t kApSmem = (size_t)kApStages * kApStage + kStateBytes +
                           kApStages * kApTok * sizeof(float) + 256;
static_assert(kStSmem <= 232448, "state kernel exceeds the shared-memory limit");
static_assert(kApSmem <= 232448, "apply kernel exceeds the shared-memory limit");

struct Plan {
    int Tk, Tq;
    Split st, ap;
};

Plan make_plan(int BH, int N, int num_sms) {
    Plan pl;
    pl.Tk = (N + kStTok - 1) / kStTok;
    pl.Tq = (N + kApTok - 1) / kApTok;
    const long long us = (long long)BH * pl.Tk, ua = (long long)BH * pl.Tq;
    pl.st = Split{us, (int)(us < num_sms ? us : num_sms)};
    pl.ap = Split{ua, (int)(ua < num_sms ? ua : num_sms)};
    return pl;
}

// Workspace: per-head counters, then the partial slots, then (for the whole
// forward) the heads' states.
size_t counters_bytes(int BH) { return ((size_t)BH * 8 + 1023) & ~size_t(1023); }
size_t partial_bytes(int BH, int N, int num_sms) {
    const Plan pl = make_plan(BH, N, num_sms);
    return ((size_t)pl.st.G + BH) * kPartialFloats * sizeof(float);
}

std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch() {
    uint32_t e = g_epoch.fetch_add(1) + 1;
    if (e == 0) e = g_epoch.fetch_add(1) + 1;   // 0 is the tag of never-used counters
    return e;
}

template <typename Kernel>
cudaError_t set_smem(Kernel k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Opt-in shared memory is a per-device attribute of a kernel.
cudaError_t configure(int dev) {
    static bool done[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    cudaError_t e;
    if ((e = set_smem(tc_state_kernel<false>, kStSmem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_state_kernel<true>, kStSmem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_apply_kernel<false>, kApSmem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_apply_kernel<true>, kApSmem)) != cudaSuccess) return e;
    done[dev] = true;
    return cudaSuccess;
}

cudaError_t launch_state(const void* k, const void* v, int BH, int N, const RopeView* rope,
                         void* workspace, uint8_t* state, unsigned* status, int num_sms,
                         cudaStream_t stream) {
    const Plan pl = make_plan(BH, N, num_sms);
    CUtensorMap mk, mv;
    if (!make_map(&mk, k, N, BH, kStTok) || !make_map(&mv, v, N, BH, kStTok))
        return cudaErrorInvalidValue;
    StateParams sp{};
    sp.N = N;
    sp.Tk = pl.Tk;
    sp.split = pl.st;
    sp.counters = reinterpret_cast<unsigned long long*>(workspace);
    sp.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counters_bytes(BH));
    sp.state = state;
    sp.epoch = next_epoch();
    sp.status = status;
    if (rope) {
        sp.rope = *rope;
        tc_state_kernel<true><<<pl.st.G, kStThreads, kStSmem, stream>>>(mk, mv, sp);
    } else {
        tc_state_kernel<false><<<pl.st.G, kStThreads, kStSmem, stream>>>(mk, mv, sp);
    }
    return cudaGetLastError();
}

cudaError_t launch_apply(const void* q, const void* g, const uint8_t* state, void* out, int BH,
                         int N, const RopeView* rope, float eps, unsigned* status, int num_sms,
                         bool after_state, cudaStream_t stream) {
    const Plan pl = make_plan(BH, N, num_sms);
    CUtensorMap mq, mg, mo;
    if (!make_map(&mq, q, N, BH, kApTok) || !make_map(&mg, g, N, BH, kApTok) ||
        !make_map(&mo, out, N, BH, kApTok))
        return cudaErrorInvalidValue;
    ApplyParams ap{};
    ap.N = N;
    ap.Tq = pl.Tq;
    ap.split = pl.ap;
    ap.state = state;
    ap.eps = eps;
    ap.status = status;
    if (rope) ap.rope = *rope;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.ap.G);
    cfg.blockDim = dim3(kApThreads);
    cfg.dynamicSmemBytes = kApSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // Only right after our own state kernel: Q and G are then complete before
    // this grid starts, whatever wrote them.
    cfg.attrs = attr;
    cfg.numAttrs = after_state ? 1 : 0;
    if (rope) return cudaLaunchKernelEx(&cfg, tc_apply_kernel<true>, mq, mg, mo, ap);
    return cudaLaunchKernelEx(&cfg, tc_apply_kernel<false>, mq, mg, mo, ap);
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

}  // namespace

size_t tc_state_workspace_bytes(int BH, int N, int num_sms) {
    return counters_bytes(BH) + partial_bytes(BH, N, num_sms);
}

size_t tc_workspace_bytes(int BH, int N, int num_sms) {
    return tc_state_workspace_bytes(BH, N, num_sms) + (size_t)BH * kStateBytes;
}

size_t tc_state_bytes(int BH) { return (size_t)BH * kStateBytes; }

cudaError_t launch_tc_state(const void* k, const void* v, void* state, int B, int H, int N,
                            const RopeView* rope, void* workspace, unsigned* status, int num_sms,
                            cudaStream_t stream) {
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    return launch_state(k, v, B * H, N, rope, workspace, static_cast<uint8_t*>(state), status,
                        num_sms, stream);
}

cudaError_t launch_tc_apply(const void* q, const void* g, const void* state, void* out, int B,
                            int H, int N, const RopeView* rope, float eps, unsigned* status,
                            int num_sms, cudaStream_t stream) {
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    return launch_apply(q, g, static_cast<const uint8_t*>(state), out, B * H, N, rope, eps,
                        status, num_sms, false, stream);
}

cudaError_t launch_tc_bf16(const void* q, const void* k, const void* v, const void* g, void* out,
                           int B, int H, int N, const RopeView* rope, float eps, float* workspace,
                           unsigned* status, int num_sms, cudaStream_t stream) {
    const int BH = B * H;
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    uint8_t* state =
        reinterpret_cast<uint8_t*>(workspace) + tc_state_workspace_bytes(BH, N, num_sms);
    if ((e = launch_state(k, v, BH, N, rope, workspace, state, status, num_sms, stream)) !=
        cudaSuccess)
        return e;
    return launch_apply(q, g, state, out, BH, N, rope, eps, status, num_sms, true, stream);
}

}  // namespace sla
