// bf16 path of the linear-attention forward on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Two persistent launches, each splitting its work units evenly over at most
// one CTA per SM ("stream-K": a CTA's range of units may cross a head):
//
//   tc_state_kernel   units = (head, 64-token tile).  Per tile the transform
//                     warps apply phi = ReLU (and the 3D RoPE) to the K tile
//                     in shared memory, in place, and accumulate
//                     z = sum phi(k) (unrotated) in registers; one thread
//                     issues S += phi~(K)^T V on the tensor core (M = N = 128,
//                     K = 64 tokens, both operands MN-major).  When a CTA
//                     leaves a head it writes its partial (S^T, z) in fp32 to
//                     workspace slot (cta + head).
//   tc_apply_kernel   units = (head, 128-token tile).  On entering a head the
//                     transform warps sum the head's partial slots into a bf16
//                     copy of S (the B operand) and z.  Per tile they apply
//                     phi/RoPE to the Q tile in place and form
//                     den = phi(q) . z + eps; one thread issues
//                     num = phi~(Q) S (M = N = K = 128) into one of two TMEM
//                     accumulators; the epilogue warps read num from TMEM,
//                     compute sigmoid(g) * num / den over the G tile in place
//                     and store it with TMA.
//
// Every mbarrier wait gives up after about a second (status word + early
// return), and every exit path waits for the copies and MMAs it issued.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

using namespace ptx;

constexpr int kRowBytes = kHeadDim * 2;          // one bf16 token row: 256 B
// A partial slot: S^T [128][128], then z as four 128-float parts (one per
// transform warp), all fp32.
constexpr int kPartialFloats = kHeadDim * kHeadDim + 4 * kHeadDim;

// ---- state kernel geometry
constexpr int kStTok = 64;                        // tokens per tile
constexpr int kStStages = 6;
constexpr int kStHalf = kStTok * 128;             // one 64-column box: 8 KB
constexpr int kStTile = 2 * kStHalf;              // one tensor tile: 16 KB
constexpr int kStStage = 2 * kStTile;             // K + V: 32 KB
constexpr int kStThreads = 192;                   // TMA warp, MMA warp, 4 transform warps
constexpr int kStTmemCols = 256;                  // two 128-column accumulators

// ---- apply kernel geometry
constexpr int kApTok = 128;
constexpr int kApStages = 3;
constexpr int kApHalf = kApTok * 128;             // 16 KB
constexpr int kApTile = 2 * kApHalf;              // 32 KB
constexpr int kApStage = 2 * kApTile;             // Q + G: 64 KB
constexpr int kApThreads = 320;                   // TMA, MMA, 4 transform, 4 epilogue warps
constexpr int kApTmemCols = 256;

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
    int N, Tk;                 // tokens per head, 64-token tiles per head
    Split split;
    RopeView rope;
    float* partial;            // slot (cta + head), kPartialFloats each
    unsigned* status;
};

struct ApplyParams {
    int N, Tq, Tk;
    Split split;               // this kernel's units: (head, 128-token tile)
    Split state_split;         // the state kernel's split, to find a head's slots
    RopeView rope;
    const float* partial;
    float eps;
    unsigned* status;
};

__device__ __forceinline__ uint32_t relu_bf2(uint32_t x) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&x);
    h = __hmax2(h, __floats2bfloat162_rn(0.f, 0.f));
    return *reinterpret_cast<uint32_t*>(&h);
}

// Rotates the pair held in one bf16x2 word by (c, s); returns the rounded pair.
__device__ __forceinline__ uint32_t rotate_bf2(uint32_t x, float2 cs) {
    float2 f = bf2_to_f2(x);
    rotate_pair(f.x, f.y, cs);
    return f2_to_bf2(f.x, f.y);
}

// Moves a grid position forward by `step` tokens (row-major t, h, w).
__device__ __forceinline__ void advance_pos(TokenPos& p, const RopeView& r, int step) {
    p.w += step;
    while (p.w >= r.Ws) {
        p.w -= r.Ws;
        if (++p.h == r.Hs) {
            p.h = 0;
            ++p.t;
        }
    }
}

// A wait taken by all 32 lanes of a warp: the warp proceeds only if every
// lane saw the phase complete, so the lanes never split on an abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// Offset of 16-byte chunk c (dims 8c..8c+7) of row r in a 128-byte-swizzled
// tile made of two 64-column boxes of `half` bytes each.
__device__ __forceinline__ uint32_t sw128_off(int r, int c, int half) {
    return (uint32_t)((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
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
    uint64_t* mma_done = accempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = p.split.start(cta), u1 = p.split.start(cta + 1);
    const uint32_t smem0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&kready[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;    // the swizzled tiles need 1 KB alignment
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
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
        // ------------------------------------------------ transform + epilogue
        const int tt = threadIdx.x - 64;          // 0..127
        const int c = tt & 15, rg = tt >> 4;       // chunk (dims 8c..8c+7), row group
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
        float zacc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
        long long it = 0;
        int seg = -1, cur_h = -1;
        bool ok = !*abort_flag;

        auto flush = [&](int sg, int hh) -> bool {
            // S^T and z of this CTA's share of head hh -> slot (cta + hh)
            if (!warp_wait(&accfull[sg & 1], (sg >> 1) & 1, abort_flag, p.status)) return false;
            tc_fence_after();
            float* slot = p.partial + (size_t)(cta + hh) * kPartialFloats;
            const int m = 32 * quad + lane;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(sg & 1) * 128 +
                              ch * 32,
                          r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    slot[(size_t)(ch * 32 + j) * kHeadDim + m] = __uint_as_float(r[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[sg & 1]);
            // lanes l and l^16 hold the same dims for neighbouring row groups
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 16);
            if (lane < 16) {
                float* zs = slot + kHeadDim * kHeadDim + (warp - 2) * kHeadDim + c * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) zs[j] = zacc[j];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
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
            TokenPos pos{};
            if (ROPE) pos = token_pos(p.rope, min(n0 + rg, p.N - 1));
#pragma unroll 2
            for (int i = 0; i < kStTok / 8; ++i) {
                const int r = rg + 8 * i;
                const uint32_t addr = kb + sw128_off(r, c, kStHalf);
                uint4 x = lds128(addr);
                x.x = relu_bf2(x.x);
                x.y = relu_bf2(x.y);
                x.z = relu_bf2(x.z);
                x.w = relu_bf2(x.w);
                const float2 f0 = bf2_to_f2(x.x), f1 = bf2_to_f2(x.y), f2 = bf2_to_f2(x.z),
                             f3 = bf2_to_f2(x.w);
                zacc[0] += f0.x; zacc[1] += f0.y; zacc[2] += f1.x; zacc[3] += f1.y;
                zacc[4] += f2.x; zacc[5] += f2.y; zacc[6] += f3.x; zacc[7] += f3.y;
                if (ROPE) {
                    if (n0 + r < p.N) {
                        x.x = rotate_bf2(x.x, rope_cs(p.rope, pos, 4 * c + 0));
                        x.y = rotate_bf2(x.y, rope_cs(p.rope, pos, 4 * c + 1));
                        x.z = rotate_bf2(x.z, rope_cs(p.rope, pos, 4 * c + 2));
                        x.w = rotate_bf2(x.w, rope_cs(p.rope, pos, 4 * c + 3));
                    }
                    advance_pos(pos, p.rope, 8);
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

__device__ __forceinline__ float gate_sigmoid(float g) {
    return __fdividef(1.f, 1.f + __expf(-g));
}

template <bool ROPE>
__global__ void __launch_bounds__(kApThreads, 1)
tc_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o, ApplyParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sbuf = smem + kApStages * kApStage;               // S^T as bf16, B operand
    float* zs = reinterpret_cast<float*>(sbuf + kApTile);       // [128]
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
            mbar_init(&qready[s], 4);
            mbar_init(&empty[s], 1);
            mbar_init(&ogather[s], 4);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], 4);
        }
        mbar_init(sready, 4);
        mbar_init(sfree, 1);
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
            long long it = 0;
            for (long long u = u0; u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
                const int s = (int)(it % kApStages);
                const uint32_t round = (uint32_t)(it / kApStages);
                if (!mbar_wait(&empty[s], (round & 1) ^ 1, abort_flag, p.status)) break;
                uint8_t* st = smem + s * kApStage;
                mbar_arrive_expect_tx(&full[s], kApStage);
                tma_load_3d(st, &tm_q, &full[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_q, &full[s], 64, tile * kApTok, h, policy);
                tma_load_3d(st + kApTile, &tm_g, &full[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApTile + kApHalf, &tm_g, &full[s], 64, tile * kApTok, h,
                            policy);
            }
            const long long first = it > kApStages ? it - kApStages : 0;
            for (long long j = first; j < it; ++j)
                mbar_wait_drain(&full[j % kApStages], (uint32_t)((j / kApStages) & 1));
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
                    if (cur_h >= 0) mma_commit(sfree);      // old state no longer read
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
    } else if (warp < 6) {
        // ------------------------------------------------ transform: state, phi, RoPE, den
        const int r = threadIdx.x - 64;            // the Q row (and S^T row) of this thread
        long long it = 0;
        int heads = 0, cur_h = -1;
        bool ok = !*abort_flag;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
            if (h != cur_h) {
                if (heads > 0 && !(ok = warp_wait(sfree, (heads - 1) & 1, abort_flag, p.status)))
                    break;
                // sum this head's partial slots: S^T row r -> bf16, swizzled K-major
                const int lo = p.state_split.owner((long long)h * p.Tk);
                const int hi = p.state_split.owner((long long)(h + 1) * p.Tk - 1);
                const uint32_t sb = smem_u32(sbuf);
#pragma unroll 1
                for (int kc = 0; kc < 16; ++kc) {
                    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
                    for (int c = lo; c <= hi; ++c) {
                        const float4* src = reinterpret_cast<const float4*>(
                            p.partial + (size_t)(c + h) * kPartialFloats + r * kHeadDim + kc * 8);
                        const float4 b0 = __ldg(src), b1 = __ldg(src + 1);
                        a0.x += b0.x; a0.y += b0.y; a0.z += b0.z; a0.w += b0.w;
                        a1.x += b1.x; a1.y += b1.y; a1.z += b1.z; a1.w += b1.w;
                    }
                    uint4 w;
                    w.x = f2_to_bf2(a0.x, a0.y);
                    w.y = f2_to_bf2(a0.z, a0.w);
                    w.z = f2_to_bf2(a1.x, a1.y);
                    w.w = f2_to_bf2(a1.z, a1.w);
                    sts128(sb + sw128_off(r, kc, kApHalf), w);
                }
                float zsum = 0.f;
                for (int c = lo; c <= hi; ++c) {
                    const float* zp = p.partial + (size_t)(c + h) * kPartialFloats +
                                      kHeadDim * kHeadDim + r;
                    zsum += __ldg(zp) + __ldg(zp + 128) + __ldg(zp + 256) + __ldg(zp + 384);
                }
                zs[r] = zsum;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sready);
                // all four transform warps have written S and z
                if (!(ok = warp_wait(sready, heads & 1, abort_flag, p.status))) break;
                ++heads;
                cur_h = h;
            }
            const int s = (int)(it % kApStages);
            const uint32_t round = (uint32_t)(it / kApStages);
            if (!(ok = warp_wait(&full[s], round & 1, abort_flag, p.status))) break;
            const uint32_t qb = smem0 + s * kApStage;
            const int n = tile * kApTok + r;
            const bool valid = n < p.N;
            TokenPos pos{};
            if (ROPE && valid) pos = token_pos(p.rope, n);
            float den = 0.f;
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
                const uint32_t addr = qb + sw128_off(r, c, kApHalf);
                uint4 x = lds128(addr);
                x.x = relu_bf2(x.x);
                x.y = relu_bf2(x.y);
                x.z = relu_bf2(x.z);
                x.w = relu_bf2(x.w);
                const float4 za = *reinterpret_cast<const float4*>(zs + 8 * c);
                const float4 zb = *reinterpret_cast<const float4*>(zs + 8 * c + 4);
                const float2 f0 = bf2_to_f2(x.x), f1 = bf2_to_f2(x.y), f2 = bf2_to_f2(x.z),
                             f3 = bf2_to_f2(x.w);
                den = fmaf(f0.x, za.x, den); den = fmaf(f0.y, za.y, den);
                den = fmaf(f1.x, za.z, den); den = fmaf(f1.y, za.w, den);
                den = fmaf(f2.x, zb.x, den); den = fmaf(f2.y, zb.y, den);
                den = fmaf(f3.x, zb.z, den); den = fmaf(f3.y, zb.w, den);
                if (ROPE && valid) {
                    x.x = rotate_bf2(x.x, rope_cs(p.rope, pos, 4 * c + 0));
                    x.y = rotate_bf2(x.y, rope_cs(p.rope, pos, 4 * c + 1));
                    x.z = rotate_bf2(x.z, rope_cs(p.rope, pos, 4 * c + 2));
                    x.w = rotate_bf2(x.w, rope_cs(p.rope, pos, 4 * c + 3));
                }
                sts128(addr, x);
            }
            dens[s * kApTok + r] = den + p.eps;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&qready[s]);
        }
    } else {
        // ------------------------------------------------ epilogue: gate, divide, store
        const int quad = warp & 3;
        const int r = 32 * quad + lane;            // TMEM lane = token row of the tile
        const bool storer = threadIdx.x == 192;
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
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)a * 128 + ch * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    const uint32_t addr = gb + sw128_off(r, ch * 4 + sub, kApHalf);
                    const uint4 gv = lds128(addr);
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 gf = bf2_to_f2(gw[e]);
                        const float o0 = __uint_as_float(v[sub * 8 + 2 * e]) * rden *
                                         gate_sigmoid(gf.x);
                        const float o1 = __uint_as_float(v[sub * 8 + 2 * e + 1]) * rden *
                                         gate_sigmoid(gf.y);
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
constexpr size_t kApSmem = (size_t)kApStages * kApStage + kApTile +
                           (kHeadDim + kApStages * kApTok) * sizeof(float) + 256;
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

template <bool ROPE>
cudaError_t launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                      const CUtensorMap& mg, const CUtensorMap& mo, const StateParams& sp,
                      const ApplyParams& ap, cudaStream_t stream) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tc_state_kernel<ROPE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kStSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc_apply_kernel<ROPE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kApSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    tc_state_kernel<ROPE><<<sp.split.G, kStThreads, kStSmem, stream>>>(mk, mv, sp);
    tc_apply_kernel<ROPE><<<ap.split.G, kApThreads, kApSmem, stream>>>(mq, mg, mo, ap);
    return cudaGetLastError();
}

}  // namespace

size_t tc_workspace_bytes(int BH, int N, int num_sms) {
    const Plan pl = make_plan(BH, N, num_sms);
    return ((size_t)pl.st.G + BH) * kPartialFloats * sizeof(float);
}

cudaError_t launch_tc_bf16(const void* q, const void* k, const void* v, const void* g, void* out,
                           int B, int H, int N, const RopeView* rope, float eps, float* workspace,
                           unsigned* status, int num_sms, cudaStream_t stream) {
    const int BH = B * H;
    const Plan pl = make_plan(BH, N, num_sms);
    CUtensorMap mk, mv, mq, mg, mo;
    if (!make_map(&mk, k, N, BH, kStTok) || !make_map(&mv, v, N, BH, kStTok) ||
        !make_map(&mq, q, N, BH, kApTok) || !make_map(&mg, g, N, BH, kApTok) ||
        !make_map(&mo, out, N, BH, kApTok))
        return cudaErrorInvalidValue;
    StateParams sp{};
    sp.N = N;
    sp.Tk = pl.Tk;
    sp.split = pl.st;
    sp.partial = workspace;
    sp.status = status;
    ApplyParams ap{};
    ap.N = N;
    ap.Tq = pl.Tq;
    ap.Tk = pl.Tk;
    ap.split = pl.ap;
    ap.state_split = pl.st;
    ap.partial = workspace;
    ap.eps = eps;
    ap.status = status;
    if (rope) {
        sp.rope = *rope;
        ap.rope = *rope;
        return launch_tc<true>(mk, mv, mq, mg, mo, sp, ap, stream);
    }
    return launch_tc<false>(mk, mv, mq, mg, mo, sp, ap, stream);
}

}  // namespace sla
