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
//                     head's counter; the CTAs whose ranges end in the head
//                     wait for all its counts and each sums a block of rows
//                     of the head's slots, in a fixed order, into the head's
//                     state: S^T in bf16, already in the tensor-core layout of
//                     the apply kernel's B operand, and z in fp32.  (The
//                     launch is cooperative, so those CTAs are resident.)
//   tc_apply_kernel   units = (head, 128-token tile).  Warp 0 streams Q tiles
//                     (and, once per head, the head's state with one bulk
//                     copy) and a last warp streams G tiles, each into its own
//                     3-slot ring.  Eight transform warps apply
//                     phi and RoPE to the Q tile in place and form
//                     den = phi(q) . z + eps; one thread of warp 1 issues
//                     num = phi~(Q) S (M = N = K = 128) into one of two TMEM
//                     accumulators; eight epilogue warps read num from TMEM,
//                     compute sigmoid(g) * num / den over the G tile in place
//                     and each stores its 32 x 64 block of o with TMA.
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
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include "launch.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sla {
namespace tc {

std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch() {
    uint32_t e = g_epoch.fetch_add(1) + 1;
    if (e == 0) e = g_epoch.fetch_add(1) + 1;   // 0 is the tag of never-used counters
    return e;
}

}  // namespace tc

namespace {

using namespace ptx;
using namespace tc;

struct StateParams {
    int N, Tk;                      // tokens per head, 64-token tiles per head
    Split split;
    RopeView rope;
    float* partial;                 // slot (cta + head), kPartialFloats each
    unsigned long long* counters;   // per head: (epoch << 32) | count, zero between launches
    uint8_t* state;                 // per head: kStateBytes
    uint32_t epoch;                 // distinct for every launch
    unsigned* status;
    // A "head" of this launch may be one block of a head's tokens: head hh
    // covers tokens [(hh % nb) * N + tok0, ...) of the RoPE grid.  merge = 0
    // leaves the partial slots unmerged (the block scan sums them).
    int nb, tok0, merge;
};

struct ApplyParams {
    int N, Tq;
    Split split;
    RopeView rope;
    const uint8_t* state;
    float eps;
    unsigned* status;
    int nb, tok0;                   // as in StateParams
    float* dden;                    // [heads][N]: kApTerms writes -(a . num) / den,
                                    // kApGrad reads the row weight (null: 1)
    float* dspart;                  // kApTerms: dS partial slots (cta + head), S^T layout
    float* dzpart;                  // kApGrad (null: none): sum_i w_i phi(g_i) per
                                    // slot (cta + head) and transform warp, [.][8][128]
    int wait_all;                   // launched as a dependent whose tiles, weights or
                                    // partials the preceding grid writes: every thread
                                    // waits for it before its first read ...
    int g_inputs;                   // ... but the G producer, when the G tiles are
                                    // inputs of the call (it prefetches them)
};

// =================================================================== state ==

template <bool ROPE>
__global__ void __launch_bounds__(kStThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_t, StateParams p) {
    constexpr int kStStages = StGeo<ROPE>::kStages;
    constexpr int kStStage = StGeo<ROPE>::kStage;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* zred = reinterpret_cast<float*>(smem + kStRing);   // [2][8 warps][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(zred + 2 * kStXWarps * kHeadDim);
    uint64_t* kready = full + kStStages;
    uint64_t* empty = kready + kStStages;
    uint64_t* accfull = empty + kStStages;        // [2]
    uint64_t* accempty = accfull + 2;             // [2]
    uint64_t* zready = accempty + 2;              // [2] the transform warps' z is in zred
    uint64_t* zfree = zready + 2;                 // [2] zred read by the flush warps
    uint64_t* slotdone = zfree + 2;               // a segment's slot is written
    uint64_t* lastknown = slotdone + 1;           // the head's last contributor is known
    uint64_t* mfull = lastknown + 1;              // merge: slots landed in the idle ring
    uint64_t* mfree = mfull + 1;                  // merge: slots read, ring reusable
    uint64_t* mma_done = mfree + 1;
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
            mbar_init(&accempty[a], kStFWarps);
            mbar_init(&zready[a], kStXWarps);
            mbar_init(&zfree[a], kStFWarps);
        }
        mbar_init(slotdone, kStFWarps);
        mbar_init(lastknown, 1);
        mbar_init(mfull, 1);
        mbar_init(mfree, kStFWarps);
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;    // the swizzled tiles need 1 KB alignment
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        if (ROPE && !rope_table_ok(p.rope)) {      // nothing of the table is read
            *abort_flag = 1;
            raise_status(p.status, kStatusBadTable);
        }
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (ROPE) prefetch_tmap(&tm_t);
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
            const uint64_t keep = policy_evict_last();   // the RoPE rows serve every head
            long long it = 0;
            int rope_h = -1, rope_base = 0;
            // (head uh, tile ut) of unit u, advanced without divisions
            int uh = (int)(u0 / p.Tk), ut = (int)(u0 % p.Tk);
            for (long long u = u0; u < u1; ++u, ++it, ut = ut + 1 == p.Tk ? 0 : ut + 1, uh += ut == 0) {
                const int h = uh, tile = ut;
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
                if (ROPE) {
                    if (h != rope_h) {                   // this head's first RoPE grid token
                        rope_h = h;
                        rope_base = (p.nb == 1 ? 0 : (h % p.nb) * p.N) + p.tok0;
                    }
                    tma_load_2d(st + 2 * kStTile, &tm_t, &full[s], 0, rope_base + tile * kStTok,
                                keep);
                }
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
            // (head uh, tile ut) of unit u, advanced without divisions
            int uh = (int)(u0 / p.Tk), ut = (int)(u0 % p.Tk);
            for (long long u = u0; ok && u < u1; ++u, ++it, ut = ut + 1 == p.Tk ? 0 : ut + 1, uh += ut == 0) {
                const int h = uh;
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
    } else if (warp < 2 + kStXWarps) {
        // ------------------------------------------------ transform: phi, RoPE, z
        const int tt = threadIdx.x - 64;           // 0..255
        const int c = tt & 15, rl = tt >> 4;        // chunk (dims 8c..8c+7), row lane 0..15
        const int xw = warp - 2;                    // transform warp 0..7
        float zacc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) zacc[j] = 0.f;

        // Hands this warp's z of segment sg to the flush warps through zred.
        auto hand_z = [&](int sg) -> bool {
            const int b = sg & 1;
            if (sg >= 2 && !warp_wait(&zfree[b], ((sg >> 1) - 1) & 1, abort_flag, p.status))
                return false;
            // lanes l and l^16 hold the same dims for neighbouring rows
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 16);
            if (lane < 16) {
                float4* zp = reinterpret_cast<float4*>(zred + (b * kStXWarps + xw) * kHeadDim +
                                                       c * 8);
                zp[0] = make_float4(zacc[0], zacc[1], zacc[2], zacc[3]);
                zp[1] = make_float4(zacc[4], zacc[5], zacc[6], zacc[7]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(&zready[b]);
            return true;
        };

        long long it = 0;
        int seg = -1, cur_h = -1;
        bool ok = !*abort_flag;
        // (head uh, tile ut) of unit u, advanced without divisions
        int uh = (int)(u0 / p.Tk), ut = (int)(u0 % p.Tk);
        for (long long u = u0; ok && u < u1; ++u, ++it, ut = ut + 1 == p.Tk ? 0 : ut + 1, uh += ut == 0) {
            const int h = uh;
            if (h != cur_h) {
                if (seg >= 0 && !(ok = hand_z(seg))) break;
                ++seg;
                cur_h = h;
            }
            const int s = (int)(it % kStStages);
            const uint32_t round = (uint32_t)(it / kStStages);
            if (!(ok = warp_wait(&full[s], round & 1, abort_flag, p.status))) break;
            const uint32_t kb = smem0 + s * kStStage;
            // all loads of the tile first, so their latencies overlap
            uint32_t addr[kStRowsPerThread];
            uint4 x[kStRowsPerThread];
#pragma unroll
            for (int i = 0; i < kStRowsPerThread; ++i) {
                addr[i] = kb + sw128_off(rl + 16 * i, c, kStHalf);
                x[i] = lds128(addr[i]);
            }
            float2 cs[kStRowsPerThread][4];
            if (ROPE) {
                // this chunk's (cos, sin) in each row's 256-byte RoPE row
#pragma unroll
                for (int i = 0; i < kStRowsPerThread; ++i)
                    unpack_cs(lds128(kb + 2 * kStTile + (rl + 16 * i) * 256 + c * 16), cs[i]);
            }
#pragma unroll
            for (int i = 0; i < kStRowsPerThread; ++i) {
                x[i].x = relu_bf2(x[i].x);
                x[i].y = relu_bf2(x[i].y);
                x[i].z = relu_bf2(x[i].z);
                x[i].w = relu_bf2(x[i].w);
                float f[8];
                unpack8(x[i], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) zacc[j] += f[j];
                if (ROPE) x[i] = rotate_chunk(f, cs[i]);
            }
#pragma unroll
            for (int i = 0; i < kStRowsPerThread; ++i) sts128(addr[i], x[i]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&kready[s]);
        }
        if (ok && seg >= 0) hand_z(seg);
    } else {
        // ------------------------------------------------ flush + merge
        // For every head segment of the CTA's range: S^T from TMEM and z from
        // zred into slot (cta + head), then the count; the head's last
        // contributor merges the head's slots.  The transform warps never wait
        // for any of this.
        const int ft = threadIdx.x - 32 * (2 + kStXWarps);   // 0..127
        const int quad = warp & 3;                           // TMEM lanes 32*quad..
        const int c = ft & 15, rq = ft >> 4;                 // merge: chunk, row lane 0..7
        const int h_first = (int)(u0 / p.Tk), h_last = (int)((u1 - 1) / p.Tk);
        int mbatch = 0;                                      // bulk merge batches issued

        // Writes the merged S^T rows [64*half, 64*half + 64) handled by this
        // thread (rows 64*half + rq + 8i, chunk c) from acc, as bf16.
        auto write_half = [&](uint8_t* dst, int half, const float4 (&acc)[8][2]) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int n = 64 * half + rq + 8 * i;
                uint4 w;
                w.x = f2_to_bf2(acc[i][0].x, acc[i][0].y);
                w.y = f2_to_bf2(acc[i][0].z, acc[i][0].w);
                w.z = f2_to_bf2(acc[i][1].x, acc[i][1].y);
                w.w = f2_to_bf2(acc[i][1].z, acc[i][1].w);
                *reinterpret_cast<uint4*>(dst + sw128_off(n, c, kStateHalf)) = w;
            }
        };
        auto add4 = [](float4& a, const float4& b) {
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        };
        // z of the head: the slots' z summed in slot order, eight slots' loads
        // in flight at a time.
        auto merge_z = [&](uint8_t* dst, int hh, int lo, int hi) {
            float zs = 0.f;
            for (int c0 = lo; c0 <= hi; c0 += 8) {
                float zq[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    zq[j] = c0 + j <= hi ? __ldcg(p.partial + (size_t)(c0 + j + hh) * kPartialFloats +
                                                  kHeadDim * kHeadDim + ft)
                                         : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + j <= hi) zs += zq[j];
            }
            reinterpret_cast<float*>(dst + kStateSBytes)[ft] = zs;
        };

        // The head's state from its partial slots, summed in slot order, read
        // from L2 (the ring is still in use).
        auto merge = [&](int hh, int lo, int hi) {
            uint8_t* dst = p.state + (size_t)hh * kStateBytes;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float4 acc[8][2];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i][0] = acc[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cc = lo; cc <= hi; ++cc) {
                    const float* src = p.partial + (size_t)(cc + hh) * kPartialFloats + c * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4* s4 = reinterpret_cast<const float4*>(
                            src + (64 * half + rq + 8 * i) * kHeadDim);
                        add4(acc[i][0], __ldcg(s4));
                        add4(acc[i][1], __ldcg(s4 + 1));
                    }
                }
                write_half(dst, half, acc);
            }
            merge_z(dst, hh, lo, hi);
        };

        // The same merge once the CTA's stage ring is idle: half-slots (32 KB,
        // 64 rows) come in by bulk copies, six at a time, and are summed from
        // shared memory in the same order.
        auto merge_bulk = [&](int hh, int lo, int hi) -> bool {
            constexpr int kHalfBytes = 64 * kHeadDim * 4;
            constexpr int kPerBatch = kStRing / kHalfBytes;   // 6
            uint8_t* dst = p.state + (size_t)hh * kStateBytes;
            bool ok2 = true;
#pragma unroll 1
            for (int half = 0; ok2 && half < 2; ++half) {
                float4 acc[8][2];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc[i][0] = acc[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int b0 = lo; ok2 && b0 <= hi; b0 += kPerBatch) {
                    const int cnt = min(kPerBatch, hi - b0 + 1);
                    if (ft == 0) {
                        if (mbatch == 0 ||
                            mbar_wait(mfree, (mbatch - 1) & 1, abort_flag, p.status)) {
                            mbar_arrive_expect_tx(mfull, cnt * kHalfBytes);
                            for (int j = 0; j < cnt; ++j)
                                bulk_load(smem + j * kHalfBytes,
                                          p.partial + (size_t)(b0 + j + hh) * kPartialFloats +
                                              64 * half * kHeadDim,
                                          kHalfBytes, mfull);
                        }
                    }
                    const int bi = mbatch++;
                    if (!(ok2 = warp_wait(mfull, bi & 1, abort_flag, p.status))) break;
                    for (int j = 0; j < cnt; ++j) {
                        const float* sl = reinterpret_cast<const float*>(smem + j * kHalfBytes);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4* s4 = reinterpret_cast<const float4*>(
                                sl + (rq + 8 * i) * kHeadDim + c * 8);
                            add4(acc[i][0], s4[0]);
                            add4(acc[i][1], s4[1]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(mfree);
                }
                if (ok2) write_half(dst, half, acc);
            }
            if (ok2) merge_z(dst, hh, lo, hi);
            return ok2;
        };

        // Rows [r0, r1) of the head's state from all its slots, in slot order;
        // with_z also sums z.  Several CTAs each merge a block of rows.
        auto merge_rows = [&](int hh, int lo, int hi, int r0, int r1, bool with_z) {
            uint8_t* dst = p.state + (size_t)hh * kStateBytes;
            const int tasks = (r1 - r0) * 16;                 // (row, 8-column chunk)
#pragma unroll 1
            for (int t0 = 0; t0 < tasks; t0 += 4 * 128) {
                float4 acc[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[i][0] = acc[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cc = lo; cc <= hi; ++cc) {
                    const float* src = p.partial + (size_t)(cc + hh) * kPartialFloats;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = t0 + i * 128 + ft;
                        if (t < tasks) {
                            const float4* s4 = reinterpret_cast<const float4*>(
                                src + (r0 + (t >> 4)) * kHeadDim + (t & 15) * 8);
                            add4(acc[i][0], __ldcg(s4));
                            add4(acc[i][1], __ldcg(s4 + 1));
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + i * 128 + ft;
                    if (t < tasks) {
                        uint4 w;
                        w.x = f2_to_bf2(acc[i][0].x, acc[i][0].y);
                        w.y = f2_to_bf2(acc[i][0].z, acc[i][0].w);
                        w.z = f2_to_bf2(acc[i][1].x, acc[i][1].y);
                        w.w = f2_to_bf2(acc[i][1].z, acc[i][1].w);
                        *reinterpret_cast<uint4*>(dst + sw128_off(r0 + (t >> 4), t & 15,
                                                                  kStateHalf)) = w;
                    }
                }
            }
            if (with_z) merge_z(dst, hh, lo, hi);
        };

        // merge_rows once the CTA's ring is idle: the rows [r0, r1) of every
        // slot come in by one batch of bulk copies and are summed from shared
        // memory in slot order (the same sums as merge_rows).
        auto merge_rows_bulk = [&](int hh, int lo, int hi, int r0, int r1, bool with_z) -> bool {
            const int k = hi - lo + 1;
            const int slot_bytes = (r1 - r0) * kHeadDim * 4;
            if (k * slot_bytes > kStRing) {        // not reached: m >= k - 1 mergers share rows
                merge_rows(hh, lo, hi, r0, r1, with_z);
                return true;
            }
            if (ft == 0) {
                if (mbatch == 0 || mbar_wait(mfree, (mbatch - 1) & 1, abort_flag, p.status)) {
                    mbar_arrive_expect_tx(mfull, k * slot_bytes);
                    for (int j = 0; j < k; ++j)
                        bulk_load(smem + j * slot_bytes,
                                  p.partial + (size_t)(lo + j + hh) * kPartialFloats +
                                      (size_t)r0 * kHeadDim,
                                  slot_bytes, mfull);
                }
            }
            const int bi = mbatch++;
            if (!warp_wait(mfull, bi & 1, abort_flag, p.status)) return false;
            uint8_t* dst = p.state + (size_t)hh * kStateBytes;
            const int tasks = (r1 - r0) * 16;                 // (row, 8-column chunk)
            for (int t = ft; t < tasks; t += 128) {
                float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
                const uint32_t off = smem0 + (uint32_t)((t >> 4) * kHeadDim * 4 + (t & 15) * 32);
                for (int j = 0; j < k; ++j) {
                    const uint4 x0 = lds128(off + j * slot_bytes);
                    const uint4 x1 = lds128(off + j * slot_bytes + 16);
                    add4(a0, make_float4(__uint_as_float(x0.x), __uint_as_float(x0.y),
                                         __uint_as_float(x0.z), __uint_as_float(x0.w)));
                    add4(a1, make_float4(__uint_as_float(x1.x), __uint_as_float(x1.y),
                                         __uint_as_float(x1.z), __uint_as_float(x1.w)));
                }
                uint4 w;
                w.x = f2_to_bf2(a0.x, a0.y);
                w.y = f2_to_bf2(a0.z, a0.w);
                w.z = f2_to_bf2(a1.x, a1.y);
                w.w = f2_to_bf2(a1.z, a1.w);
                *reinterpret_cast<uint4*>(dst + sw128_off(r0 + (t >> 4), t & 15, kStateHalf)) = w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mfree);
            if (with_z) merge_z(dst, hh, lo, hi);
            return true;
        };

        bool ok = !*abort_flag;
        for (int sg = 0; ok && sg <= h_last - h_first; ++sg) {
            const int hh = h_first + sg, b = sg & 1;
            if (!(ok = warp_wait(&accfull[b], (sg >> 1) & 1, abort_flag, p.status))) break;
            tc_fence_after();
            float* slot = p.partial + (size_t)(cta + hh) * kPartialFloats;
            const int m = 32 * quad + lane;
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)b * 128 + ch * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    slot[(size_t)(ch * 32 + j) * kHeadDim + m] = __uint_as_float(r[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[b]);
            if (!(ok = warp_wait(&zready[b], (sg >> 1) & 1, abort_flag, p.status))) break;
            float zsum = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < kStXWarps; ++w8) zsum += zred[(b * kStXWarps + w8) * kHeadDim + ft];
            slot[kHeadDim * kHeadDim + ft] = zsum;
            __syncwarp();
            if (lane == 0) mbar_arrive(&zfree[b]);
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(slotdone);
            // The head's contributors are CTAs lo..hi; those whose ranges end
            // in the head (lo..e_hi, at least lo when there are two or more)
            // finish together at the end of the kernel and share its merge.
            const int lo = p.split.owner((long long)hh * p.Tk);
            const int hi = p.split.owner((long long)(hh + 1) * p.Tk - 1);
            const int k = hi - lo + 1;
            const int e_hi = (p.split.start(hi + 1) - 1) / p.Tk == hh ? hi : hi - 1;
            const bool last_seg = hh == h_last;
            if (ft == 0) {
                // every flush warp's share of the slot is written: count this CTA in
                const bool done = mbar_wait(slotdone, sg & 1, abort_flag, p.status);
                int action = 0;                      // 0 none, 1 whole merge, 2 a block of rows
                if (done && p.merge) {
                    // (every flush thread fenced its rows of the slot before slotdone)
                    if (k == 1) {
                        action = 1;                  // one contributor: no count needed
                    } else {
                        count_contributor(p.counters + hh, p.epoch, p.status);
                        if (last_seg && wait_count(p.counters + hh, p.epoch, (uint32_t)k,
                                                   abort_flag, p.status))
                            action = 2;
                    }
                    __threadfence();
                }
                *last_flag = action;
                mbar_arrive(lastknown);
            }
            if (!(ok = warp_wait(lastknown, sg & 1, abort_flag, p.status))) break;
            const int action = *last_flag;
            if (action == 1) {
                __threadfence();
                // after the last segment every tile has been consumed: the ring is idle
                if (last_seg)
                    ok = merge_bulk(hh, lo, hi);
                else
                    merge(hh, lo, hi);
            } else if (action == 2) {
                __threadfence();
                const int m = e_hi - lo + 1, j = cta - lo;
                // a shared merge happens only at the CTA's last segment: the ring is idle
                ok = merge_rows_bulk(hh, lo, hi, j * kHeadDim / m, (j + 1) * kHeadDim / m, j == 0);
                // Each of the m CTAs sharing the merge counts once more after it has
                // seen all k contributors (here, after its merge, off the way to the
                // state); the one that reaches k + m returns the counter to zero, so
                // the next launch (a graph replay reuses its epoch) starts from an
                // empty count.
                if (ft == 0) {
                    unsigned long long* ctr = p.counters + hh;
                    if (count_contributor(ctr, p.epoch, p.status) == (uint32_t)(k + m))
                        atomicExch(ctr, 0ull);
                }
            }
        }
        // no bulk copy of ours may still be landing when the CTA exits
        if (ft == 0 && mbatch > 0) mbar_wait_drain(mfull, (mbatch - 1) & 1);
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

// MODE kApGate is the layer's apply.  The backward reuses the kernel with a
// head's state buffer that holds some 128 x 128 matrix S as S^T rows:
//   kApRaw    out_i = (R_i phi(x_i))^T S, the forward's numerator (g is not
//             read, nothing is gated);
// for the gate terms of the backward:
//   kApTerms  with num_i = (R_i phi(q_i))^T S, den_i and s_i = sigmoid(g_i):
//             out (a) = dout s / den, dg = dout num s (1 - s) / den (both bf16,
//             written over dout and g in the G slot and stored with TMA
//             through tm_o32 and tm_dg) and dden_i = -(a_i . num_i) / den_i
//             (fp32, p.dden); g and dout stream in together through the G
//             ring (tm_g, tm_d).  The tensor cores also accumulate dS = sum_i
//             (R_i phi(q_i)) a_i^T over each head segment of the CTA from the
//             tile's rotated q (Q slot) and a (G slot), both MN-major; the
//             epilogue writes each segment's dS into partial slot (cta + head)
//             of p.dspart;
// and for the masked gradients dq and dk:
//   kApGrad   out_i = [g_i > 0] (R_i^T (S x_i) + w_i z), with (S x_i)[m] =
//             sum_n x_i[n] S[m][n]: x is taken as it is (no feature map, no
//             rotation) and the buffer is read as an MN-major B operand; g is
//             the tensor whose feature map is differentiated (q or k, streamed
//             through the G ring in place of the gate), z the state's, w_i =
//             p.dden[row] (1 when null) and R_i the token's rotation (ROPE).
//             The epilogue reads z from the state buffer, which it releases
//             after the head's last tile.  The transform warps have no tile to
//             transform: with ROPE they move the RoPE rows of the tiles into
//             TMEM (columns 256 + 64 ds, one lane per token), up to DS tiles
//             ahead of the epilogue, which reads them beside the product.
//             Each warp takes 32 tokens x 32 words per tile by one TMA load
//             (tm_d is then the table's box map) into its 4 KB of shared
//             memory, and reads them back one token row per lane.  With
//             p.dzpart they also sum w_i phi(g_i) from the G slot before the
//             epilogue writes over it: a partial of dz per head segment and
//             warp.
template <bool ROPE, int MODE>
__global__ void __launch_bounds__(kApThreads, 1)
tc_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o32, const __grid_constant__ CUtensorMap tm_d,
                const __grid_constant__ CUtensorMap tm_dg, ApplyParams p) {
    constexpr int QS = ApGeo<MODE>::kQS, GS = ApGeo<MODE>::kGS, GT = ApGeo<MODE>::kGT;
    constexpr int DS = ApGeo<MODE>::kDS;
    // kApGrad: the Q tile is an operand as it is (no feature map, no
    // rotation), the state an MN-major B operand; the den slots carry the
    // RoPE rows in TMEM (or nothing without RoPE)
    constexpr bool kGrad = MODE == kApGrad;
    constexpr bool kTmemRope = kGrad && ROPE;
    constexpr bool kDS = MODE == kApTerms;       // dS accumulated beside the numerators
    // The G producer stores the outputs the epilogue staged in a G slot and
    // refills the slot as soon as the stores have read it (otherwise each
    // epilogue warp stores its own part and frees the previous tile's slot).
    constexpr bool kPStore = MODE == kApTerms;
    static_assert(kPStore || MODE != kApTerms, "the gate terms' two outputs go out from the producer");
    constexpr uint32_t kCols = kTmemRope || kDS ? 512 : kApTmemCols;
    constexpr uint32_t kRopeCol = 256;           // kTmemRope: [DS][64] columns of RoPE words
    constexpr uint32_t kDsCol = 256;             // kDS: [2][128] columns, one per head segment
    static_assert(!kTmemRope || kRopeCol + DS * 64 <= kCols, "TMEM columns");
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* qring = smem;                                      // [QS][32 KB]
    uint8_t* gring = smem + QS * kApTile;                       // [GS][GT]
    uint8_t* rscr = gring + GS * GT;                            // kTmemRope: [8 warps][4 KB]
    constexpr int kRScr = kTmemRope ? kApXWarps * 4096 : 0;
    uint8_t* sbuf = rscr + kRScr;                               // S^T bf16 (B operand), then z
    float* zs = reinterpret_cast<float*>(sbuf + kStateSBytes);  // [128]
    float* dens = zs + kHeadDim;                // [DS][128] phi(q) . z + eps (not kApGrad)
    constexpr int kDens = MODE == kApGrad ? 0 : DS * kApTok;
    // kApTerms: a . num over the second column half of each row, two tiles deep
    float* dpart = dens + kDens;                // [2][128]
    constexpr int kDPart = MODE == kApTerms ? 2 * kApTok : 0;
    uint64_t* qfull = reinterpret_cast<uint64_t*>(dpart + kDPart);
    uint64_t* qready = qfull + QS;       // Q tile transformed (MMA may read it)
    uint64_t* qempty = qready + QS;      // Q tile read by the MMA
    uint64_t* gfull = qempty + QS;
    uint64_t* gempty = gfull + GS;       // o stored from the G slot (kPStore: staged in it)
    uint64_t* dready = gempty + GS;      // [DS] den of a tile written
    uint64_t* dfree = dready + DS;        // [DS] den of a tile read
    uint64_t* accfull = dfree + DS;       // [2]
    uint64_t* accempty = accfull + 2;            // [2]
    uint64_t* sready = accempty + 2;
    uint64_t* sfree = sready + 1;
    uint64_t* mma_done = sfree + 1;
    uint64_t* pairdone = mma_done + 1;           // kApTerms: [2] the tile's dpart written
    uint64_t* rfull = pairdone + (MODE == kApTerms ? 2 : 0);   // kTmemRope: [8] a warp's rows landed
    uint64_t* dsfull = rfull + (kTmemRope ? kApXWarps : 0);   // kDS: [2] a segment's dS final
    uint64_t* dsfree = dsfull + (kDS ? 2 : 0);                // kDS: [2] written out
    uint64_t* gread = dsfree + (kDS ? 2 : 0);                 // kDS: [GS] a read by the MMA
    uint64_t* dzread = gread + (kDS ? GS : 0);                // kApGrad: [GS] x read for dz
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dzread + (kGrad ? GS : 0));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = p.split.start(cta), u1 = p.split.start(cta + 1);
    const uint32_t smem0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        if (MODE == kApTerms) {
            mbar_init(&pairdone[0], kApEWarps);
            mbar_init(&pairdone[1], kApEWarps);
        }
        if (kTmemRope)
            for (int w = 0; w < kApXWarps; ++w) mbar_init(&rfull[w], 1);
        if (kDS) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&dsfull[b], 1);
                mbar_init(&dsfree[b], kApEWarps);
            }
            for (int b = 0; b < GS; ++b) mbar_init(&gread[b], 1);
        }
        for (int s = 0; s < QS; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qready[s], kApXWarps);
            mbar_init(&qempty[s], 1);
        }
        for (int s = 0; s < GS; ++s) {
            mbar_init(&gfull[s], 1);
            mbar_init(&gempty[s], kApEWarps);
            if (kGrad) mbar_init(&dzread[s], kApXWarps);
        }
        for (int s = 0; s < DS; ++s) {
            mbar_init(&dready[s], kApXWarps);
            mbar_init(&dfree[s], kApEWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], kApEWarps);
        }
        mbar_init(sready, 1);
        // the state is free once its MMAs are done and every warp that reads
        // z is done with it: the transform warps (a copy in registers), or
        // with kApGrad the epilogue's (after the head's last tile)
        mbar_init(sfree, 1 + (kGrad ? kApEWarps : kApXWarps));
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        if (ROPE && !rope_table_ok(p.rope)) {      // nothing of the table is read
            *abort_flag = 1;
            raise_status(p.status, kStatusBadTable);
        }
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_o32);
        if (MODE == kApTerms) {
            prefetch_tmap(&tm_d);
            prefetch_tmap(&tm_dg);
        }
        if (kTmemRope) prefetch_tmap(&tm_d);
        // a dependent launch of ours may start its prologue (its CTAs take an
        // SM as ours leave it)
        griddep_launch_dependents();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (p.wait_all && !(p.g_inputs && warp == 2 + kApXWarps + kApEWarps)) griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------ Q producer (+ the heads' states)
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            // The first head's state is written by the preceding launch: its load
            // waits for that launch to complete, after the first Q tiles are in
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
            // A later head's state may load only once the previous state is free
            // (sfree); that load stays pending while tiles keep streaming, and is
            // issued from inside the waits for free stages.
            int pending = -1;
            uint32_t pend_parity = 0;
            auto resolve_pending = [&]() -> bool {
                if (pending < 0) return true;
                if (!mbar_wait(sfree, pend_parity, abort_flag, p.status)) return false;
                load_state(pending);
                pending = -1;
                return true;
            };
            auto wait_stage = [&](int s, uint32_t parity) -> bool {
                if (pending < 0) return mbar_wait(&qempty[s], parity, abort_flag, p.status);
                const uint64_t t0 = global_ns();
                for (uint32_t k = 0;; ++k) {
                    if (pending >= 0 && mbar_try_wait(sfree, pend_parity)) {
                        load_state(pending);
                        pending = -1;
                    }
                    if (mbar_try_wait_sleep(&qempty[s], parity, 2000)) return true;
                    if (*abort_flag) return false;
                    if ((k & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                        raise_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                        return false;
                    }
                }
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
                        if (!(ok = resolve_pending())) break;
                        pending = h;
                        pend_parity = (uint32_t)(heads - 1) & 1;
                    }
                    ++heads;
                    cur_h = h;
                }
                if (first_pending && it == QS) load_first();
                const int s = (int)(it % QS);
                const uint32_t round = (uint32_t)(it / QS);
                if (!(ok = wait_stage(s, (round & 1) ^ 1))) break;
                uint8_t* st = qring + s * kApTile;
                mbar_arrive_expect_tx(&qfull[s], kApTile);
                tma_load_3d(st, &tm_q, &qfull[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_q, &qfull[s], 64, tile * kApTok, h, policy);
            }
            if (ok && first_pending && first_h >= 0) load_first();
            if (ok) resolve_pending();
            // every copy issued has landed before the CTA may exit
            const long long first = it > QS ? it - QS : 0;
            for (long long j = first; j < it; ++j)
                mbar_wait_drain(&qfull[j % QS], (uint32_t)((j / QS) & 1));
            if (loads > 0) mbar_wait_drain(sready, (loads - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, false, kGrad);
            const uint32_t sb = smem_u32(sbuf);
            long long it = 0;
            int heads = 0, cur_h = -1;
            bool ok = !*abort_flag;
            // kDS: dS of tile j once the epilogue has staged its a; frees the
            // tile's Q slot and, for the producer, its G slot
            int dseg = -1;
            auto issue_ds = [&](long long j) -> bool {
                const long long uj = u0 + j;
                const int hj = (int)(uj / p.Tq);
                const bool start = j == 0 || (int)((uj - 1) / p.Tq) != hj;
                const bool end = uj + 1 == u1 || (int)((uj + 1) / p.Tq) != hj;
                if (start) {
                    ++dseg;
                    // the buffer's segment before last is written out
                    if (dseg >= 2 &&
                        !mbar_wait(&dsfree[dseg & 1], ((dseg >> 1) - 1) & 1, abort_flag, p.status))
                        return false;
                }
                const int gsj = (int)(j % GS);
                if (!mbar_wait(&gempty[gsj], (uint32_t)((j / GS) & 1), abort_flag, p.status))
                    return false;
                tc_fence_after();
                constexpr uint32_t idesc_ds = idesc_bf16(128, 128, true, true);
                const uint32_t qb = smem0 + (uint32_t)(j % QS) * kApTile;
                const uint32_t ab = smem0 + QS * kApTile + (uint32_t)gsj * GT + kApTile;
#pragma unroll
                for (int ks = 0; ks < kApTok / 16; ++ks) {
                    // 16 tokens = two 8-row swizzle atoms; the two 64-wide
                    // halves of M (and N) sit kApHalf apart
                    const uint64_t ad = smem_desc_sw128(qb + ks * 2048, kApHalf, 1024);
                    const uint64_t bd = smem_desc_sw128(ab + ks * 2048, kApHalf, 1024);
                    mma_bf16(tmem + kDsCol + (uint32_t)(dseg & 1) * 128, ad, bd, idesc_ds,
                             (start && ks == 0) ? 0u : 1u);
                }
                mma_commit(&qempty[j % QS]);
                mma_commit(&gread[gsj]);
                if (end) mma_commit(&dsfull[dseg & 1]);
                return true;
            };
            // num of tile i (its waits passed)
            auto issue_num = [&](long long i) {
                const int s = (int)(i % QS);
                const int a = (int)(i & 1);
                tc_fence_after();
                const uint32_t qb = smem0 + s * kApTile;
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                    // K-major, 128-byte swizzle: 16 k-values = 32 bytes inside a row
                    const uint32_t off = (ks >> 2) * kApHalf + (ks & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(qb + off, 16, 1024);
                    // K-major: the buffer's rows are N; MN-major: its rows are K
                    // (16 rows = 2048 bytes a step, the two N halves kStateHalf apart)
                    const uint64_t bd = kGrad
                                            ? smem_desc_sw128(sb + ks * 2048, kStateHalf, 1024)
                                            : smem_desc_sw128(sb + off, 16, 1024);
                    mma_bf16(tmem + (uint32_t)a * 128, ad, bd, idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(&accfull[a]);
            };
            if constexpr (kDS) {
                // num of tile nn and dS of tile nd < nn in whichever order their
                // inputs are ready: a tile's dS goes out as soon as its a is staged,
                // which frees its Q and G slots for the loads two tiles ahead
                // (behind the next num it would hold both rings a tile longer)
                const long long T = u1 - u0;
                long long nn = 0, nd = 0;
                int nh = (int)(u0 / p.Tq), ntile = (int)(u0 % p.Tq);   // of unit u0 + nn
                int dtile = ntile;                                      // of unit u0 + nd
                bool released = false;
                uint64_t last = global_ns();
                while (ok && nd < T) {
                    bool progress = false;
                    if (nn < T) {
                        if (nh != cur_h) {
                            if (heads > 0 && !released) {
                                mma_commit(sfree);         // old state no longer read
                                released = true;
                            }
                            if (mbar_test_wait(sready, heads & 1)) {
                                ++heads;
                                cur_h = nh;
                                released = false;
                                progress = true;
                            }
                        }
                        const int s = (int)(nn % QS), a = (int)(nn & 1);
                        const uint32_t round = (uint32_t)(nn / QS), around = (uint32_t)(nn >> 1);
                        if (nh == cur_h && mbar_test_wait(&accempty[a], (around & 1) ^ 1) &&
                            mbar_test_wait(&qready[s], round & 1) &&
                            mbar_test_wait(&qfull[s], round & 1)) {
                            issue_num(nn);
                            ++nn;
                            if (++ntile == p.Tq) {
                                ntile = 0;
                                ++nh;
                            }
                            progress = true;
                        }
                    }
                    if (nd < nn) {
                        // a head segment's first dS: its buffer's segment before last
                        // is written out
                        const bool start = nd == 0 || dtile == 0;
                        const int sg = dseg + (start ? 1 : 0);
                        if ((!start || sg < 2 ||
                             mbar_test_wait(&dsfree[sg & 1], (uint32_t)(((sg >> 1) - 1) & 1))) &&
                            mbar_test_wait(&gempty[nd % GS], (uint32_t)((nd / GS) & 1))) {
                            if (!(ok = issue_ds(nd))) break;
                            ++nd;
                            if (++dtile == p.Tq) dtile = 0;
                            progress = true;
                        }
                    }
                    if (progress) {
                        last = global_ns();
                    } else if (*abort_flag) {
                        ok = false;
                    } else if (global_ns() - last > kWaitLimitNs) {
                        raise_status(p.status, kStatusTimeout);
                        *abort_flag = 1;
                        ok = false;
                    } else {
                        __nanosleep(32);
                    }
                }
            } else {
                for (long long u = u0; ok && u < u1; ++u, ++it) {
                    const int h = (int)(u / p.Tq);
                    if (h != cur_h) {
                        if (heads > 0) mma_commit(sfree);      // old state no longer read
                        ok = mbar_wait(sready, heads & 1, abort_flag, p.status);
                        if (!ok) break;
                        ++heads;
                        cur_h = h;
                    }
                    const int s = (int)(it % QS);
                    const uint32_t round = (uint32_t)(it / QS);
                    const int a = (int)(it & 1);
                    const uint32_t around = (uint32_t)(it >> 1);
                    // (kApGrad: the tile is multiplied as it landed)
                    ok = mbar_wait(&accempty[a], (around & 1) ^ 1, abort_flag, p.status) &&
                         (kGrad || mbar_wait(&qready[s], round & 1, abort_flag, p.status)) &&
                         mbar_wait(&qfull[s], round & 1, abort_flag, p.status);
                    if (!ok) break;
                    issue_num(it);
                    mma_commit(&qempty[s]);               // the Q slot may be refilled
                }
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0);
        }
    } else if (kGrad && warp < 2 + kApXWarps) {
        // ------------------------------------------------ kApGrad: RoPE rows to TMEM, dz
        // ROPE: this warp's 32 tokens (its TMEM lanes) x 32 words of their
        // RoPE rows, by TMA to its 4 KB, then one token row per lane to TMEM.
        // p.dzpart: w_i phi(g_i) summed over rows rl + 16 i, dims 8c.., from
        // the G slot.
        const int xw = warp - 2, tquad = warp & 3, part = xw >> 2;
        const int tt = threadIdx.x - 64, c = tt & 15, rl = tt >> 4;
        uint8_t* scr = rscr + xw * 4096;
        const uint32_t scr_a = smem_u32(scr);
        uint64_t* bar = &rfull[xw];
        const uint64_t keep = policy_evict_last();
        auto issue = [&](long long u) {
            if (lane == 0) {
                const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
                const int row0 = (p.nb == 1 ? 0 : (h % p.nb) * p.N) + p.tok0 + tile * kApTok +
                                 32 * tquad;
                mbar_arrive_expect_tx(bar, 4096);
                tma_load_2d(scr, &tm_d, bar, 32 * part, row0, keep);
            }
        };
        const bool dz = p.dzpart != nullptr;
        float wnext[kApRowsPerThread], zacc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
        // the rows' weights, one tile ahead (rows past N weigh nothing)
        auto load_w = [&](long long u) {
            const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
#pragma unroll
            for (int i = 0; i < kApRowsPerThread; ++i) {
                const int row = tile * kApTok + rl + 16 * i;
                wnext[i] = row < p.N ? (p.dden ? __ldg(p.dden + (size_t)h * p.N + row) : 1.f) : 0.f;
            }
        };
        bool ok = !*abort_flag;
        long long issued = 0;
        if (ok && u0 < u1) {
            if (ROPE) {
                issue(u0);
                issued = 1;
            }
            if (dz) load_w(u0);
        }
        long long it = 0;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            uint32_t wv[32];
            if constexpr (ROPE) {
                if (!(ok = warp_wait(bar, (uint32_t)(it & 1), abort_flag, p.status))) break;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 x = lds128(scr_a + lane * 128 + ((cc ^ (lane & 7)) << 4));
                    wv[4 * cc] = x.x;
                    wv[4 * cc + 1] = x.y;
                    wv[4 * cc + 2] = x.z;
                    wv[4 * cc + 3] = x.w;
                }
                // every lane's reads are done before the next tile's copy lands there
                fence_proxy_async_smem();
                __syncwarp();
                if (u + 1 < u1) {
                    issue(u + 1);
                    ++issued;
                }
            }
            const int ds = (int)(it % DS);
            const uint32_t dround = (uint32_t)(it / DS);
            // the epilogue has read the slot's previous tile
            if (dround > 0 && !(ok = warp_wait(&dfree[ds], (dround - 1) & 1, abort_flag, p.status)))
                break;
            if constexpr (ROPE) {
                tmem_st32(tmem + ((uint32_t)(32 * tquad) << 16) + kRopeCol + (uint32_t)ds * 64 +
                              32 * part,
                          wv);
                tmem_st_wait();
                tc_fence_before();
            }
            // the epilogue may start on the tile (its RoPE rows are in TMEM); with
            // dz it writes over the G slot only once this warp has read it (dzread)
            __syncwarp();
            if (lane == 0) mbar_arrive(&dready[ds]);
            if (dz) {
                // the G slot's tile, read before the epilogue writes over it
                const int h = (int)(u / p.Tq);
                const int gs = (int)(it % GS);
                float w[kApRowsPerThread];
#pragma unroll
                for (int i = 0; i < kApRowsPerThread; ++i) w[i] = wnext[i];
                if (u + 1 < u1) load_w(u + 1);
                if (!(ok = warp_wait(&gfull[gs], (uint32_t)(it / GS) & 1, abort_flag, p.status)))
                    break;
                const uint32_t gb = smem0 + QS * kApTile + (uint32_t)gs * GT;
#pragma unroll
                for (int b4 = 0; b4 < kApRowsPerThread; b4 += 4) {
                    uint4 x[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[i] = lds128(gb + sw128_off(rl + 16 * (b4 + i), c, kApHalf));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float f[8];
                        unpack8(x[i], f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) zacc[j] = fmaf(w[b4 + i], fmaxf(f[j], 0.f), zacc[j]);
                    }
                }
                // the head segment's last tile: this warp's partial of dz
                if (u + 1 == u1 || (int)((u + 1) / p.Tq) != h) {
                    // lanes l and l ^ 16 hold the same dims for neighbouring rows
#pragma unroll
                    for (int j = 0; j < 8; ++j) zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 16);
                    if (lane < 16) {
                        float4* zp = reinterpret_cast<float4*>(
                            p.dzpart + ((size_t)(cta + h) * kApXWarps + xw) * kHeadDim + c * 8);
                        zp[0] = make_float4(zacc[0], zacc[1], zacc[2], zacc[3]);
                        zp[1] = make_float4(zacc[4], zacc[5], zacc[6], zacc[7]);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&dzread[gs]);
            }
        }
        // no copy of ours may still be landing when the CTA exits
        if (ROPE && lane == 0 && issued > it) mbar_wait_drain(bar, (uint32_t)((issued - 1) & 1));
    } else if (warp < 2 + kApXWarps) {
        // ------------------------------------------------ transform: phi, RoPE, den
        const int tt = threadIdx.x - 64;            // 0..255
        const int c = tt & 15, rl = tt >> 4;         // chunk, row lane 0..15
        float zc[8];
        // This thread's 16 bytes of the RoPE rows of its 8 rows in the next
        // tile, loaded while the current tile is transformed.
        uint4 trow[kApRowsPerThread];
        const uint64_t keep = policy_evict_last();  // the table serves every head
        // (tile `tile` of head hh; head hh is block hh % nb of its head's
        // tokens, which start at RoPE grid token (hh % nb) * N + tok0)
        auto fetch_rows = [&](int hh, int tile, int i0) {
            const int base = (p.nb == 1 ? 0 : (hh % p.nb) * p.N) + p.tok0;
#pragma unroll
            for (int i = i0; i < i0 + 4; ++i) {
                const int n = min(tile * kApTok + rl + 16 * i, p.N - 1);   // rows past N are zero
                trow[i] = ldg_nc_na128_hint(p.rope.tok + (size_t)(base + n) * kPairs + c * 4, keep);
            }
        };
        if (ROPE && u0 < u1 && !*abort_flag) {
            fetch_rows((int)(u0 / p.Tq), (int)(u0 % p.Tq), 0);
            fetch_rows((int)(u0 / p.Tq), (int)(u0 % p.Tq), 4);
        }
        long long it = 0;
        int heads = 0, cur_h = -1;
        bool ok = !*abort_flag;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tq);
            const int next_tile = u + 1 < u1 ? (int)((u + 1) % p.Tq) : -1;
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
            const int s = (int)(it % QS);
            const uint32_t round = (uint32_t)(it / QS);
            const int ds = (int)(it % DS);
            const uint32_t dround = (uint32_t)(it / DS);
            if (!(ok = warp_wait(&qfull[s], round & 1, abort_flag, p.status))) break;
            // the epilogue has read the den slot's previous tile
            if (dround > 0 && !(ok = warp_wait(&dfree[ds], (dround - 1) & 1, abort_flag, p.status)))
                break;
            const uint32_t qb = smem0 + s * kApTile;
            {
            // two batches of four rows; in each, all loads first
#pragma unroll
            for (int b4 = 0; b4 < kApRowsPerThread; b4 += 4) {
                float den[4];
                uint32_t addr[4];
                uint4 x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    addr[i] = qb + sw128_off(rl + 16 * (b4 + i), c, kApHalf);
                    x[i] = lds128(addr[i]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[i].x = relu_bf2(x[i].x);
                    x[i].y = relu_bf2(x[i].y);
                    x[i].z = relu_bf2(x[i].z);
                    x[i].w = relu_bf2(x[i].w);
                    float f[8];
                    unpack8(x[i], f);
                    if constexpr (MODE != kApRaw) {     // (the raw product has no den)
                        float2 d2 = mul2(make_float2(f[0], f[1]), make_float2(zc[0], zc[1]));
#pragma unroll
                        for (int j = 2; j < 8; j += 2)
                            d2 = fma2(make_float2(f[j], f[j + 1]), make_float2(zc[j], zc[j + 1]),
                                      d2);
                        den[i] = d2.x + d2.y;
                    }
                    if (ROPE) {
                        float2 cs[4];
                        unpack_cs(trow[b4 + i], cs);
                        x[i] = rotate_chunk(f, cs);
                    }
                }
                // rows 0-3 of the RoPE table are used: load the next tile's.  The
                // fence below waits for this thread's loads in flight, so rows 4-7
                // are loaded only after it.
                // the next unit is tile 0 of the next head, or the next tile of this one
                if (ROPE && next_tile >= 0 && b4 == 0)
                    fetch_rows(next_tile == 0 ? h + 1 : h, next_tile, 0);
#pragma unroll
                for (int i = 0; i < 4; ++i) sts128(addr[i], x[i]);
                if constexpr (MODE == kApRaw) continue;
                // Sum den over the 16 chunk lanes of each row: each step halves the
                // rows a lane holds, so lane c ends with row b4 + ((c >> 2) & 3).
                const bool b3 = (c >> 3) & 1, b2 = (c >> 2) & 1;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float send = b3 ? den[k] : den[k + 2];
                    const float keep = b3 ? den[k + 2] : den[k];
                    den[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                    const float send = b2 ? den[0] : den[1];
                    const float keep = b2 ? den[1] : den[0];
                    den[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                den[0] += __shfl_xor_sync(0xffffffffu, den[0], 2);
                den[0] += __shfl_xor_sync(0xffffffffu, den[0], 1);
                if ((c & 3) == 0)
                    dens[ds * kApTok + rl + 16 * (b4 + ((c >> 2) & 3))] = den[0] + p.eps;
            }
            fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&qready[s]);
                mbar_arrive(&dready[ds]);
            }
            if (ROPE && next_tile >= 0) fetch_rows(next_tile == 0 ? h + 1 : h, next_tile, 4);
        }
    } else if (warp < 2 + kApXWarps + kApEWarps) {
        // ------------------------------------------------ epilogue: gate, divide, store
        const int ew = warp - 2 - kApXWarps;        // 0..7
        const int quad = warp & 3, hf = ew >> 2;     // TMEM lanes 32*quad.., columns 64*hf..
        const int r = 32 * quad + lane;              // TMEM lane = token row of the tile
        long long it = 0;
        int eheads = 0, ecur_h = -1;                 // kApGrad: heads begun
        int eseg = 0;                                // kDS: head segments written out
        bool ok = !*abort_flag;
        for (long long u = u0; ok && u < u1; ++u, ++it) {
            const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
            const int gs = (int)(it % GS);
            const uint32_t ground = (uint32_t)(it / GS);
            const int ds = (int)(it % DS);
            const int a = (int)(it & 1);
            const uint32_t around = (uint32_t)(it >> 1);
            // kApGrad: the row's weight, loaded before the waits (rows past N
            // are not stored: any row serves)
            float w = 1.f;
            if constexpr (MODE == kApGrad) {
                if (p.dden) w = p.dden[(size_t)h * p.N + min(tile * kApTok + r, p.N - 1)];
            }
            ok = warp_wait(&accfull[a], around & 1, abort_flag, p.status) &&
                 warp_wait(&dready[ds], (uint32_t)(it / DS) & 1, abort_flag, p.status) &&
                 warp_wait(&gfull[gs], ground & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const float den = kGrad ? 1.f : dens[ds * kApTok + r];   // (kApGrad: none)
            const float inv_den = 1.f / den;
            float part = 0.f;
            // (with the RoPE rows in the slot's TMEM columns, the slot is
            // freed after the chunks)
            if constexpr (!kGrad) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&dfree[ds]);
            }
            if constexpr (MODE == kApGrad) {
                if (h != ecur_h) {
                    // the head's state has landed (sready) and stays until this
                    // warp, among others, is done with its z (sfree)
                    if (!(ok = warp_wait(sready, eheads & 1, abort_flag, p.status))) break;
                    ++eheads;
                    ecur_h = h;
                }
            }
            const uint32_t gb = smem0 + QS * kApTile + gs * GT;
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t addr[4];
                uint4 gv[4];
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    addr[sub] = gb + sw128_off(r, hf * 8 + ch * 4 + sub, kApHalf);
                    if (MODE != kApRaw) gv[sub] = lds128(addr[sub]);
                }
                uint4 dv[4];                          // kApTerms: dout, in the stage's second tile
                if constexpr (MODE == kApTerms) {
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) dv[sub] = lds128(addr[sub] + kApTile);
                }
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)a * 128 + hf * 64 +
                              ch * 32,
                          v);
                uint32_t csw[16];                     // kTmemRope: the chunk's 16 pairs
                if constexpr (kTmemRope)
                    tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + kRopeCol + (uint32_t)ds * 64 +
                                  32 * hf + 16 * ch,
                              csw);
                tmem_ld_wait();
                if constexpr (MODE == kApTerms) {
                    // a over dout, dg over g; part collects a . num of the row
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        uint4 av;
                        terms_chunk(gv[sub], dv[sub], v + 8 * sub, inv_den, av, gv[sub], part);
                        sts128(addr[sub] + kApTile, av);
                    }
                } else if constexpr (MODE == kApGate) {
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) gv[sub] = gate_chunk(gv[sub], v + 8 * sub, den);
                } else if constexpr (MODE == kApGrad) {
                    const float* zw = zs + 64 * hf + ch * 32;
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        uint4 cs = {};
                        if constexpr (kTmemRope)
                            cs = make_uint4(csw[4 * sub], csw[4 * sub + 1], csw[4 * sub + 2],
                                            csw[4 * sub + 3]);
                        gv[sub] = grad_chunk<ROPE>(gv[sub], v + 8 * sub, cs, w, zw + 8 * sub);
                    }
                    // with dz, the transform warps read x from the slot: the first
                    // write over it waits for them
                    if (ch == 0 && p.dzpart &&
                        !(ok = warp_wait(&dzread[gs], ground & 1, abort_flag, p.status)))
                        break;
                } else {
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        const uint32_t* n8 = v + 8 * sub;
                        gv[sub] = make_uint4(
                            f2_to_bf2(__uint_as_float(n8[0]), __uint_as_float(n8[1])),
                            f2_to_bf2(__uint_as_float(n8[2]), __uint_as_float(n8[3])),
                            f2_to_bf2(__uint_as_float(n8[4]), __uint_as_float(n8[5])),
                            f2_to_bf2(__uint_as_float(n8[6]), __uint_as_float(n8[7])));
                    }
                }
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) sts128(addr[sub], gv[sub]);
            }
            if (!ok) break;
            tc_fence_before();
            fence_proxy_async_smem();
            if constexpr (kGrad) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&dfree[ds]);
            }
            if constexpr (MODE == kApGrad) {
                // the head's last tile here: its state may be replaced
                if (u + 1 == u1 || (int)((u + 1) / p.Tq) != h) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sfree);
                }
            }
            if constexpr (MODE == kApTerms) {
                // dden of the row from the two column halves (the warp of the
                // other half has the same rows)
                const int pb = (int)(it & 1);
                if (hf == 1) dpart[pb * kApTok + r] = part;
                __syncwarp();
                if (lane == 0) mbar_arrive(&pairdone[pb]);
                if (!(ok = warp_wait(&pairdone[pb], (uint32_t)(it >> 1) & 1, abort_flag,
                                     p.status)))
                    break;
                const int row = tile * kApTok + r;
                if (hf == 0 && row < p.N)
                    p.dden[(size_t)h * p.N + row] = -(part + dpart[pb * kApTok + r]) * inv_den;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&accempty[a]);
                if constexpr (kPStore) {
                    mbar_arrive(&gempty[gs]);       // this warp's part is staged (a, dg)
                } else {
                    // this warp's rows 32*quad.. of column half hf, 4 KB of the tile
                    tma_store_3d(&tm_o32, gring + gs * GT + hf * kApHalf + quad * kApORows * 128,
                                 64 * hf, tile * kApTok + quad * kApORows, h);
                    bulk_commit();
                    // the previous tile's store has read its G slot, which may be refilled
                    bulk_wait_read_one();
                    if (it > 0) mbar_arrive(&gempty[(it - 1) % GS]);
                }
            }
            if constexpr (kDS) {
                // the head segment's last tile here: its dS (rows r of S^T's
                // columns, as the state kernel's slots hold them) to slot cta + h
                if (u + 1 == u1 || (int)((u + 1) / p.Tq) != h) {
                    const int sb = eseg & 1;
                    if (!(ok = warp_wait(&dsfull[sb], (uint32_t)(eseg >> 1) & 1, abort_flag,
                                         p.status)))
                        break;
                    tc_fence_after();
                    float* slot = p.dspart + (size_t)(cta + h) * kPartialFloats;
#pragma unroll 1
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t v[32];
                        tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + kDsCol + (uint32_t)sb * 128 +
                                      hf * 64 + ch * 32,
                                  v);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            slot[(size_t)(hf * 64 + ch * 32 + j) * kHeadDim + r] = __uint_as_float(v[j]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dsfree[sb]);
                    ++eseg;
                }
            }
        }
        if (!kPStore && lane == 0) bulk_wait_all();
    } else {
        // ------------------------------------------------ G producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            // kPStore: the outputs of tile j, staged in its slot, go out from here
            // (kApTerms: a over the dout half, dg over the g half)
            auto store_tile = [&](long long j) -> bool {
                const long long uj = u0 + j;
                const int h = (int)(uj / p.Tq), tile = (int)(uj % p.Tq);
                const int s = (int)(j % GS);
                if (!mbar_wait(&gempty[s], (uint32_t)((j / GS) & 1), abort_flag, p.status))
                    return false;
                const uint8_t* st = gring + s * GT;
#pragma unroll 1
                for (int b = 0; b < 8; ++b) {
                    const int hf = b >> 2, quad = b & 3;
                    const uint8_t* box = st + hf * kApHalf + quad * kApORows * 128;
                    tma_store_3d(&tm_o32, box + (MODE == kApTerms ? kApTile : 0), 64 * hf,
                                 tile * kApTok + quad * kApORows, h);
                    if (MODE == kApTerms)
                        tma_store_3d(&tm_dg, box, 64 * hf, tile * kApTok + quad * kApORows, h);
                }
                bulk_commit();
                return true;
            };
            long long it = 0, stored = 0;
            bool ok = true;
            for (long long u = u0; u < u1; ++u, ++it) {
                const int h = (int)(u / p.Tq), tile = (int)(u % p.Tq);
                const int s = (int)(it % GS);
                const uint32_t round = (uint32_t)(it / GS);
                if constexpr (kPStore) {
                    // the slot's previous tile is stored and read out of it
                    if (it >= GS) {
                        if (!(ok = store_tile(it - GS))) break;
                        ++stored;
                        bulk_wait_read_all();
                        // kDS: and the MMA has read the tile's a for dS
                        if (kDS && !(ok = mbar_wait(&gread[s], (uint32_t)(((it - GS) / GS) & 1),
                                                    abort_flag, p.status)))
                            break;
                    }
                } else if (!mbar_wait(&gempty[s], (round & 1) ^ 1, abort_flag, p.status)) {
                    break;
                }
                if constexpr (MODE == kApRaw) {
                    mbar_arrive(&gfull[s]);         // the slot only stages the output
                    continue;
                }
                uint8_t* st = gring + s * GT;
                mbar_arrive_expect_tx(&gfull[s], GT);
                tma_load_3d(st, &tm_g, &gfull[s], 0, tile * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_g, &gfull[s], 64, tile * kApTok, h, policy);
                if (MODE == kApTerms) {             // dout next to g
                    tma_load_3d(st + kApTile, &tm_d, &gfull[s], 0, tile * kApTok, h, policy);
                    tma_load_3d(st + kApTile + kApHalf, &tm_d, &gfull[s], 64, tile * kApTok, h,
                                policy);
                }
            }
            // the last tiles' outputs; every store is complete before the CTA exits
            if constexpr (kPStore) {
                for (; ok && stored < it; ++stored) ok = store_tile(stored);
                bulk_wait_all();
            }
            const long long first = it > GS ? it - GS : 0;
            for (long long j = first; j < it; ++j)
                mbar_wait_drain(&gfull[j % GS], (uint32_t)((j / GS) & 1));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kCols);
    }
}

// =================================================================== fused ==
//
// One cluster of C CTAs per head does the whole forward of that head in one
// launch (for shapes with few heads per SM, where the two-launch path pays
// its fixed costs: launch, ramp, merge tail).  Phase 1: CTA r of the cluster
// streams its share of the head's K and V tiles as the state kernel does,
// accumulating its partial S^T in TMEM and its z in registers, and writes
// both to its own shared memory.  Reduction: every CTA sums the C partial z
// itself, which lets its transform warps start on its first Q tile, while
// CTA r sums rows [r*128/C, (r+1)*128/C) of the C partial S^T through
// distributed shared memory and writes them, as bf16 in the MMA layout, into
// every CTA's state buffer.  Phase 2: CTA r applies the state to its share of
// the head's Q and G tiles as the apply kernel does.  With p.state_out, CTA r
// also copies its rows of the state (and CTA 0 the head's z) to global memory,
// in the layout the state kernel writes, for a backward that reuses it.  The cluster meets only
// on mbarriers with bounded waits, and on one cluster barrier just before
// exit, which every thread reaches after bounded work.
//
// Shared memory in phase 2: the Q ring's first stage and the G ring's first
// two stages are loaded as soon as phase 1 ends; the partial S^T sits in Q
// stages 1-2 and the partial z in G stage 2, which are loaded only once every
// CTA of the cluster has read them.

constexpr int kFuThreads = kApThreads;            // the apply kernel's 19 warps
constexpr int kFuTmemCols = 512;                  // phase 2 at 0 and 128, phase 1 at 256
constexpr int kFuMaxCluster = 8;
constexpr int kFuAutoMaxTiles = 64;               // heads the shape rule always fuses
constexpr int kFuPartial = kApTile;               // partial S^T fp32 [128][128]: Q stages 1-2
constexpr int kFuZLocal = kApQStages * kApTile + 2 * kApTile;   // partial z: G stage 2
static_assert(kFuPartial + kHeadDim * kHeadDim * 4 == kApQStages * kApTile, "Q stages 1-2");
static_assert(kStXWarps * kHeadDim * 4 <= kStateSBytes, "z parts fit in the state buffer");

struct FusedParams {
    int N, Tk, Tq, C;           // tokens, 64-token and 128-token tiles per head, cluster size
    RopeView rope;
    float eps;
    unsigned* status;
    uint8_t* state_out;         // null, or the heads' states (kStateBytes each) written out
};

template <bool ROPE>
__global__ void __launch_bounds__(kFuThreads, 1)
tc_fused_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_t, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o32, FusedParams p) {
    constexpr int kS1 = StGeo<ROPE>::kStages;   // phase-1 ring
    constexpr int kS1Stage = StGeo<ROPE>::kStage;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* qring = smem;                                      // phase 2
    uint8_t* gring = smem + kApQStages * kApTile;               // phase 2
    float* partial = reinterpret_cast<float*>(smem + kFuPartial);   // S^T [128][128]
    float* zloc = reinterpret_cast<float*>(smem + kFuZLocal);       // z of this CTA [128]
    uint8_t* sbuf = smem + kStRing;                             // S^T bf16, then z
    float* zparts = reinterpret_cast<float*>(sbuf);             // [8 warps][128] before the merge
    float* zs = reinterpret_cast<float*>(sbuf + kStateSBytes);
    float* dens = zs + kHeadDim;                // [kApDSlots][128] phi(q) . z + eps
    uint64_t* full = reinterpret_cast<uint64_t*>(dens + kApDSlots * kApTok);
    uint64_t* kready = full + kS1;
    uint64_t* empty = kready + kS1;
    uint64_t* s1full = empty + kS1;          // phase-1 MMAs done: TMEM partial final, ring idle
    uint64_t* zpdone = s1full + 1;           // the transform warps' z parts written (8 warps)
    uint64_t* flushdone = zpdone + 1;        // partial S^T and z written (4 warps)
    uint64_t* pready = flushdone + 1;        // every CTA's partial written (C arrivals)
    uint64_t* zready = pready + 1;           // z of the head in zs (4 warps)
    uint64_t* reddone = zready + 1;          // this CTA's rows written everywhere (8 warps)
    uint64_t* sready = reddone + 1;          // the state is complete here (own rows, others' bytes)
    uint64_t* qfull = sready + 1;
    uint64_t* qready = qfull + kApQStages;
    uint64_t* qempty = qready + kApQStages;
    uint64_t* gfull = qempty + kApQStages;
    uint64_t* gempty = gfull + kApGStages;
    uint64_t* dready = gempty + kApGStages;
    uint64_t* dfree = dready + kApDSlots;
    uint64_t* accfull = dfree + kApDSlots;   // [2]
    uint64_t* accempty = accfull + 2;        // [2]
    uint64_t* mma_done = accempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const uint32_t rank = cluster_ctarank();
    const int h = blockIdx.x / C;                               // the head of this cluster
    const int k0 = (int)((long long)rank * p.Tk / C), k1 = (int)((long long)(rank + 1) * p.Tk / C);
    const int q0 = (int)((long long)rank * p.Tq / C), q1 = (int)((long long)(rank + 1) * p.Tq / C);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t tmem_acc1 = 256;          // phase-1 accumulator column

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS1; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&kready[s], kStXWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(s1full, 1);
        mbar_init(zpdone, kStXWarps);
        mbar_init(flushdone, kStFWarps);
        mbar_init(pready, C);
        mbar_init(zready, kStFWarps);
        mbar_init(reddone, kApEWarps);
        mbar_init(sready, 1);
        for (int s = 0; s < kApQStages; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qready[s], kApXWarps);
            mbar_init(&qempty[s], 1);
        }
        for (int s = 0; s < kApGStages; ++s) {
            mbar_init(&gfull[s], 1);
            mbar_init(&gempty[s], kApEWarps);
        }
        for (int s = 0; s < kApDSlots; ++s) {
            mbar_init(&dready[s], kApXWarps);
            mbar_init(&dfree[s], kApEWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], kApEWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        if (ROPE && !rope_table_ok(p.rope)) {      // nothing of the table is read
            *abort_flag = 1;
            raise_status(p.status, kStatusBadTable);
        }
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        if (ROPE) prefetch_tmap(&tm_t);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_o32);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kFuTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    // the other CTAs' barriers are initialised before anyone arrives on them
    cluster_arrive();
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ producer: K, V, then Q
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            const uint64_t keep = policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int t = k0; t < k1; ++t, ++it) {
                const int s = it % kS1;
                const uint32_t round = (uint32_t)(it / kS1);
                if (!(ok = mbar_wait(&empty[s], (round & 1) ^ 1, abort_flag, p.status))) break;
                uint8_t* st = smem + s * kS1Stage;
                mbar_arrive_expect_tx(&full[s], kS1Stage);
                tma_load_3d(st, &tm_k, &full[s], 0, t * kStTok, h, policy);
                tma_load_3d(st + kStHalf, &tm_k, &full[s], 64, t * kStTok, h, policy);
                tma_load_3d(st + kStTile, &tm_v, &full[s], 0, t * kStTok, h, policy);
                tma_load_3d(st + kStTile + kStHalf, &tm_v, &full[s], 64, t * kStTok, h, policy);
                if (ROPE) tma_load_2d(st + 2 * kStTile, &tm_t, &full[s], 0, t * kStTok, keep);
            }
            // Q stage 0 reuses the phase-1 ring once every phase-1 tile is
            // consumed; stages 1-2 hold the partial S^T until the cluster has
            // read it
            if (ok) ok = mbar_wait(s1full, 0, abort_flag, p.status);
            int jt = 0;
            for (int t = q0; ok && t < q1; ++t, ++jt) {
                const int s = jt % kApQStages;
                const uint32_t round = (uint32_t)(jt / kApQStages);
                if (jt == 1 && !(ok = mbar_wait_cluster(sready, 0, abort_flag, p.status))) break;
                if (!(ok = mbar_wait(&qempty[s], (round & 1) ^ 1, abort_flag, p.status))) break;
                uint8_t* st = qring + s * kApTile;
                mbar_arrive_expect_tx(&qfull[s], kApTile);
                tma_load_3d(st, &tm_q, &qfull[s], 0, t * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_q, &qfull[s], 64, t * kApTok, h, policy);
            }
            // every copy issued has landed before the CTA may exit
            if (jt == 0) {
                const int first = it > kS1 ? it - kS1 : 0;
                for (int j = first; j < it; ++j)
                    mbar_wait_drain(&full[j % kS1], (uint32_t)((j / kS1) & 1));
            }
            const int first = jt > kApQStages ? jt - kApQStages : 0;
            for (int j = first; j < jt; ++j)
                mbar_wait_drain(&qfull[j % kApQStages], (uint32_t)((j / kApQStages) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = !*abort_flag;
            {
                constexpr uint32_t idesc = idesc_bf16(128, 128, true, true);
                int it = 0;
                for (int t = k0; ok && t < k1; ++t, ++it) {
                    const int s = it % kS1;
                    const uint32_t round = (uint32_t)(it / kS1);
                    ok = mbar_wait(&kready[s], round & 1, abort_flag, p.status) &&
                         mbar_wait(&full[s], round & 1, abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = smem0 + s * kS1Stage, vb = kb + kStTile;
#pragma unroll
                    for (int ks = 0; ks < kStTok / 16; ++ks) {
                        const uint64_t a = smem_desc_sw128(kb + ks * 2048, kStHalf, 1024);
                        const uint64_t b = smem_desc_sw128(vb + ks * 2048, kStHalf, 1024);
                        mma_bf16(tmem + tmem_acc1, a, b, idesc, (it > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(s1full);
            }
            if (ok) ok = mbar_wait_cluster(sready, 0, abort_flag, p.status);
            if (ok) {
                fence_proxy_async_all();
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
                const uint32_t sb = smem_u32(sbuf);
                int it = 0;
                for (int t = q0; ok && t < q1; ++t, ++it) {
                    const int s = it % kApQStages;
                    const uint32_t round = (uint32_t)(it / kApQStages);
                    const int a = it & 1;
                    const uint32_t around = (uint32_t)(it >> 1);
                    ok = mbar_wait(&accempty[a], (around & 1) ^ 1, abort_flag, p.status) &&
                         mbar_wait(&qready[s], round & 1, abort_flag, p.status) &&
                         mbar_wait(&qfull[s], round & 1, abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t qb = smem0 + s * kApTile;
#pragma unroll
                    for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * kApHalf + (ks & 3) * 32;
                        const uint64_t ad = smem_desc_sw128(qb + off, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(sb + off, 16, 1024);
                        mma_bf16(tmem + (uint32_t)a * 128, ad, bd, idesc, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&accfull[a]);
                    mma_commit(&qempty[s]);
                }
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0);
        }
    } else if (warp < 2 + kApXWarps) {
        // ------------------------------------------------ transform: K (z, RoPE), then Q
        const int tt = threadIdx.x - 64;            // 0..255
        const int c = tt & 15, rl = tt >> 4;
        const int xw = warp - 2;
        bool ok = !*abort_flag;
        {
            float zacc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) zacc[j] = 0.f;
            int it = 0;
            for (int t = k0; ok && t < k1; ++t, ++it) {
                const int s = it % kS1;
                const uint32_t round = (uint32_t)(it / kS1);
                if (!(ok = warp_wait(&full[s], round & 1, abort_flag, p.status))) break;
                const uint32_t kb = smem0 + s * kS1Stage;
                uint32_t addr[kStRowsPerThread];
                uint4 x[kStRowsPerThread];
#pragma unroll
                for (int i = 0; i < kStRowsPerThread; ++i) {
                    addr[i] = kb + sw128_off(rl + 16 * i, c, kStHalf);
                    x[i] = lds128(addr[i]);
                }
                float2 cs[kStRowsPerThread][4];
                if (ROPE) {
#pragma unroll
                    for (int i = 0; i < kStRowsPerThread; ++i)
                        unpack_cs(lds128(kb + 2 * kStTile + (rl + 16 * i) * 256 + c * 16), cs[i]);
                }
#pragma unroll
                for (int i = 0; i < kStRowsPerThread; ++i) {
                    x[i].x = relu_bf2(x[i].x);
                    x[i].y = relu_bf2(x[i].y);
                    x[i].z = relu_bf2(x[i].z);
                    x[i].w = relu_bf2(x[i].w);
                    float f[8];
                    unpack8(x[i], f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) zacc[j] += f[j];
                    if (ROPE) x[i] = rotate_chunk(f, cs[i]);
                }
#pragma unroll
                for (int i = 0; i < kStRowsPerThread; ++i) sts128(addr[i], x[i]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kready[s]);
            }
            // this warp's z into the z parts (the state buffer is idle until
            // the cluster has published its partials)
            if (ok) {
#pragma unroll
                for (int j = 0; j < 8; ++j) zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 16);
                if (lane < 16) {
                    float4* zp = reinterpret_cast<float4*>(zparts + xw * kHeadDim + c * 8);
                    zp[0] = make_float4(zacc[0], zacc[1], zacc[2], zacc[3]);
                    zp[1] = make_float4(zacc[4], zacc[5], zacc[6], zacc[7]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(zpdone);
            }
        }
        // phase 2 starts as soon as z of the head is known
        if (ok) ok = warp_wait(zready, 0, abort_flag, p.status);
        float zc[8];
        if (ok) {
            const float4 za = *reinterpret_cast<const float4*>(zs + 8 * c);
            const float4 zb = *reinterpret_cast<const float4*>(zs + 8 * c + 4);
            zc[0] = za.x; zc[1] = za.y; zc[2] = za.z; zc[3] = za.w;
            zc[4] = zb.x; zc[5] = zb.y; zc[6] = zb.z; zc[7] = zb.w;
        }
        uint4 trow[kApRowsPerThread];
        const uint64_t keep = policy_evict_last();  // the table serves every head
        auto fetch_rows = [&](int tile, int i0) {
#pragma unroll
            for (int i = i0; i < i0 + 4; ++i) {
                const int n = min(tile * kApTok + rl + 16 * i, p.N - 1);
                trow[i] = ldg_nc_na128_hint(p.rope.tok + (size_t)n * kPairs + c * 4, keep);
            }
        };
        if (ROPE && ok && q0 < q1) {
            fetch_rows(q0, 0);
            fetch_rows(q0, 4);
        }
        int it = 0;
        for (int t = q0; ok && t < q1; ++t, ++it) {
            const int next_tile = t + 1 < q1 ? t + 1 : -1;
            const int s = it % kApQStages;
            const uint32_t round = (uint32_t)(it / kApQStages);
            const int ds = it % kApDSlots;
            const uint32_t dround = (uint32_t)(it / kApDSlots);
            if (!(ok = warp_wait(&qfull[s], round & 1, abort_flag, p.status))) break;
            if (dround > 0 && !(ok = warp_wait(&dfree[ds], (dround - 1) & 1, abort_flag, p.status)))
                break;
            const uint32_t qb = smem0 + s * kApTile;
#pragma unroll
            for (int b4 = 0; b4 < kApRowsPerThread; b4 += 4) {
                float den[4];
                uint32_t addr[4];
                uint4 x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    addr[i] = qb + sw128_off(rl + 16 * (b4 + i), c, kApHalf);
                    x[i] = lds128(addr[i]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    x[i].x = relu_bf2(x[i].x);
                    x[i].y = relu_bf2(x[i].y);
                    x[i].z = relu_bf2(x[i].z);
                    x[i].w = relu_bf2(x[i].w);
                    float f[8];
                    unpack8(x[i], f);
                    float2 d2 = mul2(make_float2(f[0], f[1]), make_float2(zc[0], zc[1]));
#pragma unroll
                    for (int j = 2; j < 8; j += 2)
                        d2 = fma2(make_float2(f[j], f[j + 1]), make_float2(zc[j], zc[j + 1]), d2);
                    den[i] = d2.x + d2.y;
                    if (ROPE) {
                        float2 cs[4];
                        unpack_cs(trow[b4 + i], cs);
                        x[i] = rotate_chunk(f, cs);
                    }
                }
                if (ROPE && next_tile >= 0 && b4 == 0) fetch_rows(next_tile, 0);
#pragma unroll
                for (int i = 0; i < 4; ++i) sts128(addr[i], x[i]);
                const bool b3 = (c >> 3) & 1, b2 = (c >> 2) & 1;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float send = b3 ? den[k] : den[k + 2];
                    const float keep = b3 ? den[k + 2] : den[k];
                    den[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                }
                {
                    const float send = b2 ? den[0] : den[1];
                    const float keep = b2 ? den[1] : den[0];
                    den[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
                den[0] += __shfl_xor_sync(0xffffffffu, den[0], 2);
                den[0] += __shfl_xor_sync(0xffffffffu, den[0], 1);
                if ((c & 3) == 0)
                    dens[ds * kApTok + rl + 16 * (b4 + ((c >> 2) & 3))] = den[0] + p.eps;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&qready[s]);
                mbar_arrive(&dready[ds]);
            }
            if (ROPE && next_tile >= 0) fetch_rows(next_tile, 4);
        }
    } else if (warp < 2 + kApXWarps + kApEWarps) {
        // ------------------------------------------------ flush, reduction, epilogue
        const int ew = warp - 2 - kApXWarps;        // 0..7
        const int quad = warp & 3, hf = ew >> 2;
        const int rt = threadIdx.x - 32 * (2 + kApXWarps);   // 0..255
        bool ok = !*abort_flag;
        const uint32_t pbase = smem_u32(partial), zbase = smem_u32(zloc), sbase = smem_u32(sbuf);
        // phase 1 (four of the warps): the partial S^T from TMEM, and the sum
        // of the eight z parts, into shared memory
        if (ew < kStFWarps) {
            if (ok) ok = warp_wait(s1full, 0, abort_flag, p.status);
            if (ok) {
                tc_fence_after();
                const int m = 32 * quad + lane;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + tmem_acc1 + ch * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        partial[(ch * 32 + j) * kHeadDim + m] = __uint_as_float(r[j]);
                }
                tc_fence_before();
            }
            if (ok) ok = warp_wait(zpdone, 0, abort_flag, p.status);
            if (ok) {
                float z = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < kStXWarps; ++w8) z += zparts[w8 * kHeadDim + rt];
                zloc[rt] = z;
                __syncwarp();
                if (lane == 0) mbar_arrive(flushdone);
            }
        }
        // every warp of this CTA has written its share: tell the cluster
        // (each arrive releases at cluster scope what this thread has seen
        // through flushdone: the other warps' partial rows and z)
        if (rt == 0 && ok && mbar_wait(flushdone, 0, abort_flag, p.status)) {
            for (int q = 0; q < C; ++q) mbar_arrive_cluster(mapa_shared(smem_u32(pready), q));
        }
        if (ok) ok = warp_wait_cluster(pready, 0, abort_flag, p.status);
        // z of the head first (the transform warps wait for it), every CTA's
        // part loaded before any is added, added in rank order
        if (ok && ew < kStFWarps) {
            float zq[kFuMaxCluster];
#pragma unroll
            for (int q = 0; q < kFuMaxCluster; ++q)
                if (q < C) zq[q] = ld_cluster_f32(mapa_shared(zbase + rt * 4, q));
            float z = 0.f;
#pragma unroll
            for (int q = 0; q < kFuMaxCluster; ++q)
                if (q < C) z += zq[q];
            zs[rt] = z;
            if (p.state_out) fence_proxy_async_smem();   // z is read by a bulk copy
            __syncwarp();
            if (lane == 0) mbar_arrive(zready);
        }
        // rows [rank*128/C, (rank+1)*128/C) of S^T, summed in rank order from
        // every CTA's partial (four CTAs' loads in flight at a time), written as
        // bf16 into this CTA's state buffer and pushed from there to the others
        if (ok) {
            const int r0 = (int)rank * kHeadDim / C, r1 = ((int)rank + 1) * kHeadDim / C;
            const int tasks = (r1 - r0) * 16;
            for (int t = rt; t < tasks; t += 32 * kApEWarps) {
                const int n = r0 + (t >> 4), cc = t & 15;
                const uint32_t off = (uint32_t)((n * kHeadDim + cc * 8) * 4);
                float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
                for (int qb = 0; qb < C; qb += 4) {
                    float4 b0[4], b1[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (qb + j < C) {
                            const uint32_t src = mapa_shared(pbase + off, qb + j);
                            b0[j] = ld_cluster_f4(src);
                            b1[j] = ld_cluster_f4(src + 16);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (qb + j < C) {
                            a0.x += b0[j].x; a0.y += b0[j].y; a0.z += b0[j].z; a0.w += b0[j].w;
                            a1.x += b1[j].x; a1.y += b1[j].y; a1.z += b1[j].z; a1.w += b1[j].w;
                        }
                    }
                }
                uint4 w;
                w.x = f2_to_bf2(a0.x, a0.y);
                w.y = f2_to_bf2(a0.z, a0.w);
                w.z = f2_to_bf2(a1.x, a1.y);
                w.w = f2_to_bf2(a1.z, a1.w);
                sts128(sbase + sw128_off(n, cc, kStateHalf), w);
            }
            fence_proxy_async_smem();                    // the rows are read by bulk copies
            __syncwarp();
            if (lane == 0) mbar_arrive(reddone);
            if (rt == 0 && mbar_wait(reddone, 0, abort_flag, p.status)) {
                // the rows are contiguous in each 64-column half of the buffer; a
                // CTA's state is complete when its own rows are written (this
                // arrival) and the other CTAs' rows have landed (their bytes)
                const uint32_t rows = (uint32_t)(r1 - r0) * 128;
                for (int q = 0; q < C; ++q) {
                    if (q == (int)rank) continue;
                    const uint32_t bar = mapa_shared(smem_u32(sready), q);
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t off = (uint32_t)hh * kStateHalf + (uint32_t)r0 * 128;
                        bulk_push_cluster(mapa_shared(sbase + off, q), sbase + off, rows, bar);
                    }
                }
                if (p.state_out) {
                    // the same rows to the head's state in global memory, and z from
                    // CTA 0 (this thread is one of z's writers; it waits for the rest)
                    uint8_t* dst = p.state_out + (size_t)h * kStateBytes;
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t off = (uint32_t)hh * kStateHalf + (uint32_t)r0 * 128;
                        bulk_store(dst + off, sbase + off, rows);
                    }
                    if (rank == 0 && mbar_wait(zready, 0, abort_flag, p.status))
                        bulk_store(dst + kStateSBytes, smem_u32(zs), kHeadDim * 4);
                }
                bulk_commit();
                mbar_arrive_expect_tx(sready, (uint32_t)(kHeadDim - (r1 - r0)) * 256);
                bulk_wait_read_all();                    // (before the CTA may exit)
            }
        }
        // phase 2: the epilogue of the apply kernel
        if (ok) ok = warp_wait_cluster(sready, 0, abort_flag, p.status);
        const int r = 32 * quad + lane;
        int it = 0;
        for (int t = q0; ok && t < q1; ++t, ++it) {
            const int gs = it % kApGStages;
            const uint32_t ground = (uint32_t)(it / kApGStages);
            const int ds = it % kApDSlots;
            const int a = it & 1;
            const uint32_t around = (uint32_t)(it >> 1);
            ok = warp_wait(&accfull[a], around & 1, abort_flag, p.status) &&
                 warp_wait(&dready[ds], (uint32_t)(it / kApDSlots) & 1, abort_flag, p.status) &&
                 warp_wait(&gfull[gs], ground & 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const float den = dens[ds * kApTok + r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&dfree[ds]);
            const uint32_t gb = smem0 + kApQStages * kApTile + gs * kApTile;
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t addr[4];
                uint4 gv[4];
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    addr[sub] = gb + sw128_off(r, hf * 8 + ch * 4 + sub, kApHalf);
                    gv[sub] = lds128(addr[sub]);
                }
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)a * 128 + hf * 64 +
                              ch * 32,
                          v);
                tmem_ld_wait();
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) gv[sub] = gate_chunk(gv[sub], v + 8 * sub, den);
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) sts128(addr[sub], gv[sub]);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&accempty[a]);
                tma_store_3d(&tm_o32, gring + gs * kApTile + hf * kApHalf + quad * kApORows * 128,
                             64 * hf, t * kApTok + quad * kApORows, h);
                bulk_commit();
                bulk_wait_read_one();
                if (it > 0) mbar_arrive(&gempty[(it - 1) % kApGStages]);
            }
        }
        if (lane == 0) bulk_wait_all();
    } else {
        // ------------------------------------------------ G producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t policy = policy_evict_first();
            // stages 0-1 are free once phase 1 is done; stage 2 holds this
            // CTA's partial z until the cluster has read it
            bool ok = mbar_wait(s1full, 0, abort_flag, p.status);
            int it = 0;
            for (int t = q0; ok && t < q1; ++t, ++it) {
                const int s = it % kApGStages;
                const uint32_t round = (uint32_t)(it / kApGStages);
                if (it == 2 && !(ok = mbar_wait_cluster(sready, 0, abort_flag, p.status))) break;
                if (!(ok = mbar_wait(&gempty[s], (round & 1) ^ 1, abort_flag, p.status))) break;
                uint8_t* st = gring + s * kApTile;
                mbar_arrive_expect_tx(&gfull[s], kApTile);
                tma_load_3d(st, &tm_g, &gfull[s], 0, t * kApTok, h, policy);
                tma_load_3d(st + kApHalf, &tm_g, &gfull[s], 64, t * kApTok, h, policy);
            }
            const int first = it > kApGStages ? it - kApGStages : 0;
            for (int j = first; j < it; ++j)
                mbar_wait_drain(&gfull[j % kApGStages], (uint32_t)((j / kApGStages) & 1));
        }
    }

    tc_fence_before();
    __syncthreads();
    // no CTA leaves while another may still read or write its shared memory
    cluster_arrive();
    cluster_wait();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kFuTmemCols);
    }
}

// ========================================================== block scan ==
//
// Block-causal form: the state kernel runs over (head, block) segments and
// leaves each segment's partial slots unmerged; this kernel turns them into
// running states.  For head h it starts from the incoming carried state (or
// zero), adds block b's slots in slot order and writes the running sum as the
// bf16 state of segment (h, b) for the apply kernel, for b = 0, 1, ...; the
// final sum is the outgoing carried state.  The running sum stays in fp32.
//
// CTA (h, r) owns rows [16 r, 16 r + 16) of S^T (value dims); thread t adds
// row 16 r + t/16, key dims 8 (t % 16) .. +7.  CTA (h, 0) also carries z.

constexpr int kScanRows = 16;
constexpr int kScanThreads = kScanRows * 16;      // one thread per (row, 8 key dims)
constexpr int kScanBatch = 4;                     // slots whose loads are in flight at once

struct ScanParams {
    const float* partial;       // the state kernel's slots (cta + segment)
    Split split;                // the state kernel's split over segments
    int Tk, nb;                 // 64-token tiles per segment, blocks per head
    const float* state_in;      // [heads][128*128 + 128]: S[m][n], then z; or null
    float* state_out;           // same layout, or null (may equal state_in)
    uint8_t* states;            // [heads*nb][kStateBytes]
};

__global__ void __launch_bounds__(kScanThreads)
block_scan_kernel(ScanParams p) {
    griddep_wait();                       // the slots are complete
    griddep_launch_dependents();          // the apply kernel may start its prologue
    const int head = blockIdx.x, rg = blockIdx.y, t = threadIdx.x;
    const int n = kScanRows * rg + (t >> 4), cc = t & 15;
    const bool with_z = rg == 0 && t < kHeadDim;
    constexpr int kCarried = kHeadDim * kHeadDim + kHeadDim;
    float acc[8], z = 0.f;
    if (p.state_in) {
        const float* sin = p.state_in + (size_t)head * kCarried;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = sin[(cc * 8 + j) * kHeadDim + n];
        if (with_z) z = sin[kHeadDim * kHeadDim + t];
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    }
    for (int b = 0; b < p.nb; ++b) {
        const int sh = head * p.nb + b;
        const int lo = p.split.owner((long long)sh * p.Tk);
        const int hi = p.split.owner((long long)(sh + 1) * p.Tk - 1);
        // the block's slots, kScanBatch loaded before any is added, added in order
        for (int c0 = lo; c0 <= hi; c0 += kScanBatch) {
            float4 x0[kScanBatch], x1[kScanBatch];
            float zx[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) {
                if (c0 + j <= hi) {
                    const float* slot = p.partial + (size_t)(c0 + j + sh) * kPartialFloats;
                    const float4* src = reinterpret_cast<const float4*>(slot + n * kHeadDim + cc * 8);
                    x0[j] = __ldcg(src);
                    x1[j] = __ldcg(src + 1);
                    zx[j] = with_z ? __ldcg(slot + kHeadDim * kHeadDim + t) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) {
                if (c0 + j <= hi) {
                    acc[0] += x0[j].x; acc[1] += x0[j].y; acc[2] += x0[j].z; acc[3] += x0[j].w;
                    acc[4] += x1[j].x; acc[5] += x1[j].y; acc[6] += x1[j].z; acc[7] += x1[j].w;
                    z += zx[j];
                }
            }
        }
        uint8_t* dst = p.states + (size_t)sh * kStateBytes;
        uint4 w;
        w.x = f2_to_bf2(acc[0], acc[1]);
        w.y = f2_to_bf2(acc[2], acc[3]);
        w.z = f2_to_bf2(acc[4], acc[5]);
        w.w = f2_to_bf2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(dst + sw128_off(n, cc, kStateHalf)) = w;
        if (with_z) reinterpret_cast<float*>(dst + kStateSBytes)[t] = z;
    }
    if (p.state_out) {
        float* sout = p.state_out + (size_t)head * kCarried;
#pragma unroll
        for (int j = 0; j < 8; ++j) sout[(cc * 8 + j) * kHeadDim + n] = acc[j];
        if (with_z) sout[kHeadDim * kHeadDim + t] = z;
    }
}

// The backward's dS state from the apply kernel's partials: for every head,
// the dS^T slots (cta + head) of the CTAs whose range holds the head's query
// tiles, summed in CTA order as bf16 rows in the MMA layout, and z from the
// slots' per-warp partials (warp order within a CTA).
struct DsMergeParams {
    const float* dspart;        // [slots][kPartialFloats] (the z part unused)
    const float* dzpart;        // [slots][8 warps][128]
    uint8_t* states;            // [heads][kStateBytes]
    Split split;                // the apply kernel's units (head, 128-token tile)
    int Tq;
};

__global__ void __launch_bounds__(kScanThreads)
ds_merge_kernel(DsMergeParams p) {
    // (launched as a programmatic dependent: the partials are complete after this)
    griddep_wait();
    griddep_launch_dependents();
    const int head = blockIdx.x, rg = blockIdx.y, t = threadIdx.x;
    const int n = kScanRows * rg + (t >> 4), cc = t & 15;
    const bool with_z = rg == 0 && t < kHeadDim;
    const int lo = p.split.owner((long long)head * p.Tq);
    const int hi = p.split.owner((long long)(head + 1) * p.Tq - 1);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c0 = lo; c0 <= hi; c0 += kScanBatch) {
        float4 x0[kScanBatch], x1[kScanBatch];
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (c0 + j <= hi) {
                const float4* src = reinterpret_cast<const float4*>(
                    p.dspart + (size_t)(c0 + j + head) * kPartialFloats + n * kHeadDim + cc * 8);
                x0[j] = __ldcg(src);
                x1[j] = __ldcg(src + 1);
            }
        }
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
            if (c0 + j <= hi) {
                acc[0] += x0[j].x; acc[1] += x0[j].y; acc[2] += x0[j].z; acc[3] += x0[j].w;
                acc[4] += x1[j].x; acc[5] += x1[j].y; acc[6] += x1[j].z; acc[7] += x1[j].w;
            }
        }
    }
    uint8_t* dst = p.states + (size_t)head * kStateBytes;
    uint4 w;
    w.x = f2_to_bf2(acc[0], acc[1]);
    w.y = f2_to_bf2(acc[2], acc[3]);
    w.z = f2_to_bf2(acc[4], acc[5]);
    w.w = f2_to_bf2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(dst + sw128_off(n, cc, kStateHalf)) = w;
    if (with_z) {
        float z = 0.f;
        for (int c = lo; c <= hi; ++c) {
            const float* zp = p.dzpart + (size_t)(c + head) * kApXWarps * kHeadDim + t;
            float x[kApXWarps];
#pragma unroll
            for (int w8 = 0; w8 < kApXWarps; ++w8) x[w8] = __ldcg(zp + w8 * kHeadDim);
#pragma unroll
            for (int w8 = 0; w8 < kApXWarps; ++w8) z += x[w8];
        }
        reinterpret_cast<float*>(dst + kStateSBytes)[t] = z;
    }
}

// ==================================================================== host ==

// Barriers and flags follow the buffers: state 3*stages + 13 mbarriers plus
// three words, apply 3*Q stages + 2*G stages + 2*den slots + 7 mbarriers plus
// two words.
template <bool ROPE>
constexpr size_t st_smem() {
    return (size_t)kStRing + 2 * kStXWarps * kHeadDim * sizeof(float) +
           (3 * StGeo<ROPE>::kStages + 13) * 8 + 16;
}
template <bool ROPE, int MODE = kApGate>
constexpr size_t ap_smem() {
    using G = ApGeo<MODE>;
    constexpr bool kTmemRope = MODE == kApGrad && ROPE;
    return (size_t)G::kQS * kApTile + (size_t)G::kGS * G::kGT + (kTmemRope ? kApXWarps * 4096 : 0) +
           kStateBytes +
           ((MODE == kApGrad ? 0 : G::kDS) + (MODE == kApTerms ? 2 : 0)) * kApTok * sizeof(float) +
           (3 * G::kQS + 2 * G::kGS + 2 * G::kDS + 7 + (MODE == kApTerms ? 2 + 4 + G::kGS : 0) +
            (MODE == kApGrad ? G::kGS : 0) + (kTmemRope ? kApXWarps : 0)) *
               8 +
           16;
}
// fused: the ring, the state, the denominators, then 3*stages + 7 phase-1 and
// cluster mbarriers, the apply kernel's 3*Q + 2*G + 2*den + 5 and two words.
template <bool ROPE>
constexpr size_t fu_smem() {
    return (size_t)kStRing + kStateBytes + kApDSlots * kApTok * sizeof(float) +
           (3 * StGeo<ROPE>::kStages + 7 + 3 * kApQStages + 2 * kApGStages + 2 * kApDSlots + 5) *
               8 +
           16;
}
static_assert(fu_smem<true>() <= 232448 && fu_smem<false>() <= 232448, "fused kernel smem");
static_assert(st_smem<true>() <= 232448 && st_smem<false>() <= 232448, "state kernel smem");
static_assert(ap_smem<true>() <= 232448 && ap_smem<false>() <= 232448, "apply kernel smem");
static_assert(ap_smem<true, kApTerms>() <= 232448, "apply kernel smem, gate terms");
static_assert(ap_smem<true, kApGrad>() <= 232448, "apply kernel smem, masked gradient");
static_assert(ap_smem<true, kApRaw>() <= 232448, "apply kernel smem, raw product");

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

template <typename Kernel>
cudaError_t set_smem(Kernel k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Opt-in shared memory is a per-device attribute of a kernel.  The entry points
// call this under locks of their own (the workspace's, the fixed array's), so it
// takes one of its own too.
cudaError_t configure(int dev) {
    static std::atomic<bool> done[64] = {};
    static std::mutex mu;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    cudaError_t e;
    if ((e = set_smem(tc_state_kernel<false>, st_smem<false>())) != cudaSuccess) return e;
    if ((e = set_smem(tc_state_kernel<true>, st_smem<true>())) != cudaSuccess) return e;
    if ((e = set_smem(tc_apply_kernel<false, kApGate>, ap_smem<false>())) != cudaSuccess) return e;
    if ((e = set_smem(tc_apply_kernel<true, kApGate>, ap_smem<true>())) != cudaSuccess) return e;
    if ((e = set_smem(tc_apply_kernel<false, kApRaw>, ap_smem<false, kApRaw>())) != cudaSuccess)
        return e;
    if ((e = set_smem(tc_apply_kernel<true, kApRaw>, ap_smem<true, kApRaw>())) != cudaSuccess)
        return e;
    if ((e = set_smem(tc_apply_kernel<false, kApTerms>, ap_smem<false, kApTerms>())) !=
        cudaSuccess)
        return e;
    if ((e = set_smem(tc_apply_kernel<true, kApTerms>, ap_smem<true, kApTerms>())) != cudaSuccess)
        return e;
    if ((e = set_smem(tc_apply_kernel<false, kApGrad>, ap_smem<false, kApGrad>())) != cudaSuccess)
        return e;
    if ((e = set_smem(tc_apply_kernel<true, kApGrad>, ap_smem<true, kApGrad>())) != cudaSuccess)
        return e;
    if ((e = set_smem(tc_fused_kernel<false>, fu_smem<false>())) != cudaSuccess) return e;
    if ((e = set_smem(tc_fused_kernel<true>, fu_smem<true>())) != cudaSuccess) return e;
    done[dev].store(true, std::memory_order_release);
    return cudaSuccess;
}

// BH "heads" of N tokens; in the block-causal form each is one block of nb
// per head, starting at token tok0 of the RoPE grid, and merge is 0.
cudaError_t launch_state(const void* k, const void* v, int BH, int N, const RopeView* rope,
                         void* workspace, uint8_t* state, unsigned* status, int num_sms,
                         cudaStream_t stream, int nb = 1, int tok0 = 0, bool merge = true) {
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
    sp.nb = nb;
    sp.tok0 = tok0;
    sp.merge = merge ? 1 : 0;
    CUtensorMap mt = mk;   // without RoPE the table map is never read
    if (rope && !make_rope_map(&mt, rope->tok, rope->need, kStTok)) return cudaErrorInvalidValue;
    if (rope) sp.rope = *rope;
    // Cooperative: all CTAs are resident together, which the shared merge of a
    // head's state relies on (its CTAs wait for each other's counts).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.st.G);
    cfg.blockDim = dim3(kStThreads);
    cfg.dynamicSmemBytes = rope ? st_smem<true>() : st_smem<false>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (rope) return cudaLaunchKernelEx(&cfg, tc_state_kernel<true>, mk, mv, mt, sp);
    return cudaLaunchKernelEx(&cfg, tc_state_kernel<false>, mk, mv, mt, sp);
}

cudaError_t launch_apply(const void* q, const void* g, const uint8_t* state, void* out, int BH,
                         int N, const RopeView* rope, float eps, unsigned* status, int num_sms,
                         int pdl, cudaStream_t stream, int nb = 1, int tok0 = 0,
                         int mode = kApGate, const void* dout = nullptr, void* dg = nullptr,
                         float* dden = nullptr, float* dspart = nullptr, float* dzpart = nullptr) {
    const Plan pl = make_plan(BH, N, num_sms);
    CUtensorMap mq, mg, mo;
    if (!make_map(&mq, q, N, BH, kApTok) || !make_map(&mg, g, N, BH, kApTok) ||
        !make_map(&mo, out, N, BH, kApORows))
        return cudaErrorInvalidValue;
    CUtensorMap md = mg, mdg = mo;     // read and written only by the gate terms
    if (mode == kApTerms &&
        (!make_map(&md, dout, N, BH, kApTok) || !make_map(&mdg, dg, N, BH, kApORows)))
        return cudaErrorInvalidValue;
    // the masked gradient with RoPE: md is the table's box map
    if (mode == kApGrad && rope && !make_rope_box_map(&md, rope->tok, rope->need))
        return cudaErrorInvalidValue;
    ApplyParams ap{};
    ap.N = N;
    ap.Tq = pl.Tq;
    ap.split = pl.ap;
    ap.state = state;
    ap.eps = eps;
    ap.status = status;
    ap.nb = nb;
    ap.tok0 = tok0;
    ap.dden = dden;
    ap.dspart = dspart;
    ap.dzpart = dzpart;
    ap.wait_all = pdl == kPdlWaitAll || pdl == kPdlWaitAllButG ? 1 : 0;
    ap.g_inputs = pdl == kPdlWaitAllButG ? 1 : 0;
    if (rope) ap.rope = *rope;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.ap.G);
    cfg.blockDim = dim3(kApThreads);
    cfg.dynamicSmemBytes =
        mode == kApTerms  ? (rope ? ap_smem<true, kApTerms>() : ap_smem<false, kApTerms>())
        : mode == kApGrad ? (rope ? ap_smem<true, kApGrad>() : ap_smem<false, kApGrad>())
        : mode == kApRaw  ? (rope ? ap_smem<true, kApRaw>() : ap_smem<false, kApRaw>())
                          : (rope ? ap_smem<true>() : ap_smem<false>());
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // A programmatic dependent only right after a kernel of ours: kPdlState when
    // that kernel writes nothing but the state (Q and G are then complete before
    // this grid starts, whatever wrote them), kPdlWaitAll otherwise.
    cfg.attrs = attr;
    cfg.numAttrs = pdl != kPdlNone ? 1 : 0;
    if (mode == kApRaw) {
        if (rope)
            return cudaLaunchKernelEx(&cfg, tc_apply_kernel<true, kApRaw>, mq, mg, mo, md, mdg, ap);
        return cudaLaunchKernelEx(&cfg, tc_apply_kernel<false, kApRaw>, mq, mg, mo, md, mdg, ap);
    }
    if (mode == kApTerms) {
        if (rope)
            return cudaLaunchKernelEx(&cfg, tc_apply_kernel<true, kApTerms>, mq, mg, mo, md, mdg, ap);
        return cudaLaunchKernelEx(&cfg, tc_apply_kernel<false, kApTerms>, mq, mg, mo, md, mdg, ap);
    }
    if (mode == kApGrad) {
        if (rope)
            return cudaLaunchKernelEx(&cfg, tc_apply_kernel<true, kApGrad>, mq, mg, mo, md, mdg, ap);
        return cudaLaunchKernelEx(&cfg, tc_apply_kernel<false, kApGrad>, mq, mg, mo, md, mdg, ap);
    }
    if (rope)
        return cudaLaunchKernelEx(&cfg, tc_apply_kernel<true, kApGate>, mq, mg, mo, md, mdg, ap);
    return cudaLaunchKernelEx(&cfg, tc_apply_kernel<false, kApGate>, mq, mg, mo, md, mdg, ap);
}

template <bool ROPE>
cudaLaunchConfig_t fused_config(int BH, int C, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BH * C);
    cfg.blockDim = dim3(kFuThreads);
    cfg.dynamicSmemBytes = fu_smem<ROPE>();
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// How many clusters of C fused CTAs the device holds at once (cached per
// device, variant and C; 0 if the query fails).
int fused_capacity(int dev, bool rope, int C) {
    static int cache[64][2][kFuMaxCluster + 1];
    static bool known[64][2][kFuMaxCluster + 1];
    static std::mutex mu;
    if (dev < 0 || dev >= 64 || C < 2 || C > kFuMaxCluster) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!known[dev][rope][C]) {
        cudaLaunchAttribute attr[1];
        int n = 0;
        cudaError_t e;
        if (rope) {
            cudaLaunchConfig_t cfg = fused_config<true>(1, C, nullptr, attr);
            e = cudaOccupancyMaxActiveClusters(&n, tc_fused_kernel<true>, &cfg);
        } else {
            cudaLaunchConfig_t cfg = fused_config<false>(1, C, nullptr, attr);
            e = cudaOccupancyMaxActiveClusters(&n, tc_fused_kernel<false>, &cfg);
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev][rope][C] = n;
        known[dev][rope][C] = true;
    }
    return cache[dev][rope][C];
}

// The forward's kernels: SLA_FORWARD_KERNEL = "fused" or "split" forces one
// (fused only where it applies), anything else lets the shape decide.
enum class Path { kAuto, kFused, kSplit };

Path forced_path() {
    const char* v = std::getenv("SLA_FORWARD_KERNEL");
    if (!v) return Path::kAuto;
    if (!std::strcmp(v, "fused")) return Path::kFused;
    if (!std::strcmp(v, "split")) return Path::kSplit;
    return Path::kAuto;
}

// The cluster size of the fused kernel for this shape, or 0 for the two
// launches.  Every head needs its own cluster resident at once (the cluster's
// CTAs wait for each other), so C is the largest size, at most 8 and at most
// the head's 128-token tiles (every CTA then has at least one tile of each
// phase), for which all B*H clusters fit on the device together.
int fused_cluster(int dev, int BH, int N, bool rope, int num_sms) {
    const Path path = forced_path();
    if (path == Path::kSplit) return 0;
    const int Tq = (N + kApTok - 1) / kApTok;
    int cmax = num_sms / BH;
    if (cmax > kFuMaxCluster) cmax = kFuMaxCluster;
    if (cmax > Tq) cmax = Tq;
    int C = cmax;
    while (C >= 2 && fused_capacity(dev, rope, C) < BH) --C;
    if (C < 2) return 0;
    // Measured on B300: the fused launch saves the second launch, the merge
    // through global memory and the hand-over between the launches, but it
    // leaves SMs idle when B*H does not divide their number.  It wins for
    // heads of up to 64 query tiles, and for longer heads only when its
    // clusters cover at least 85% of the SMs.
    if (path == Path::kAuto && Tq > kFuAutoMaxTiles && 100 * BH * C < 85 * num_sms) return 0;
    return C;
}

cudaError_t launch_fused(const void* q, const void* k, const void* v, const void* g, void* out,
                         int BH, int N, int C, const RopeView* rope, float eps, unsigned* status,
                         cudaStream_t stream, uint8_t* state_out) {
    CUtensorMap mk, mv, mq, mg, mo;
    if (!make_map(&mk, k, N, BH, kStTok) || !make_map(&mv, v, N, BH, kStTok) ||
        !make_map(&mq, q, N, BH, kApTok) || !make_map(&mg, g, N, BH, kApTok) ||
        !make_map(&mo, out, N, BH, kApORows))
        return cudaErrorInvalidValue;
    CUtensorMap mt = mk;   // without RoPE the table map is never read
    if (rope && !make_rope_map(&mt, rope->tok, N, kStTok)) return cudaErrorInvalidValue;
    FusedParams fp{};
    fp.N = N;
    fp.Tk = (N + kStTok - 1) / kStTok;
    fp.Tq = (N + kApTok - 1) / kApTok;
    fp.C = C;
    if (rope) fp.rope = *rope;
    fp.eps = eps;
    fp.status = status;
    fp.state_out = state_out;
    cudaLaunchAttribute attr[1];
    if (rope) {
        cudaLaunchConfig_t cfg = fused_config<true>(BH, C, stream, attr);
        return cudaLaunchKernelEx(&cfg, tc_fused_kernel<true>, mk, mv, mt, mq, mg, mo, fp);
    }
    cudaLaunchConfig_t cfg = fused_config<false>(BH, C, stream, attr);
    return cudaLaunchKernelEx(&cfg, tc_fused_kernel<false>, mk, mv, mt, mq, mg, mo, fp);
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

}  // namespace

size_t tc_counter_bytes(int BH) { return counters_bytes(BH); }

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
                        num_sms, stream, 1, 0, true);
}

cudaError_t launch_tc_apply(const void* q, const void* g, const void* state, void* out, int B,
                            int H, int N, const RopeView* rope, float eps, unsigned* status,
                            int num_sms, cudaStream_t stream, int mode, const void* dout,
                            void* dg, float* dden, float* dspart, float* dzpart, int pdl) {
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    return launch_apply(q, g, static_cast<const uint8_t*>(state), out, B * H, N, rope, eps,
                        status, num_sms, pdl, stream, 1, 0, mode, dout, dg, dden, dspart,
                        dzpart);
}

size_t tc_apply_partial_bytes(int BH, int N, int num_sms) {
    const Plan pl = make_plan(BH, N, num_sms);
    return ((size_t)pl.ap.G + BH) * kPartialFloats * sizeof(float);
}

size_t tc_apply_zpart_bytes(int BH, int N, int num_sms) {
    const Plan pl = make_plan(BH, N, num_sms);
    return ((size_t)pl.ap.G + BH) * kApXWarps * kHeadDim * sizeof(float);
}

cudaError_t launch_tc_ds_merge(const float* dspart, const float* dzpart, void* state, int B, int H,
                               int N, int num_sms, cudaStream_t stream, bool pdl) {
    const Plan pl = make_plan(B * H, N, num_sms);
    DsMergeParams mp{dspart, dzpart, static_cast<uint8_t*>(state), pl.ap, pl.Tq};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * H, kHeadDim / kScanRows);
    cfg.blockDim = dim3(kScanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, ds_merge_kernel, mp);
}

int tc_forward_cluster(int dev, int BH, int N, bool rope, int num_sms) {
    if (configure(dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return fused_cluster(dev, BH, N, rope, num_sms);
}

cudaError_t launch_tc_fused(const void* q, const void* k, const void* v, const void* g, void* out,
                            int B, int H, int N, int C, const RopeView* rope, float eps,
                            unsigned* status, cudaStream_t stream, void* state_out) {
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    return launch_fused(q, k, v, g, out, B * H, N, C, rope, eps, status, stream,
                        static_cast<uint8_t*>(state_out));
}

cudaError_t launch_tc_block_causal(const void* q, const void* k, const void* v, const void* g,
                                   void* out, int B, int H, int N, int block_tokens,
                                   const RopeView* rope, int rope_offset, float eps,
                                   const float* state_in, float* state_out, float* workspace,
                                   unsigned* status, int num_sms, cudaStream_t stream) {
    const int BH = B * H, nb = N / block_tokens, BHs = BH * nb;
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    uint8_t* states = reinterpret_cast<uint8_t*>(workspace) +
                      tc_state_workspace_bytes(BHs, block_tokens, num_sms);
    // the (head, block) segments' partial slots, left unmerged
    if ((e = launch_state(k, v, BHs, block_tokens, rope, workspace, nullptr, status, num_sms,
                          stream, nb, rope_offset, false)) != cudaSuccess)
        return e;
    const Plan pl = make_plan(BHs, block_tokens, num_sms);
    ScanParams sp{};
    sp.partial = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) +
                                          counters_bytes(BHs));
    sp.split = pl.st;
    sp.Tk = pl.Tk;
    sp.nb = nb;
    sp.state_in = state_in;
    sp.state_out = state_out;
    sp.states = states;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BH, kHeadDim / kScanRows);
    cfg.blockDim = dim3(kScanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, block_scan_kernel, sp)) != cudaSuccess) return e;
    return launch_apply(q, g, states, out, BHs, block_tokens, rope, eps, status, num_sms,
                        kPdlState, stream, nb, rope_offset);
}

cudaError_t launch_tc_two_phase(const void* q, const void* k, const void* v, const void* g,
                                void* out, int B, int H, int N, const RopeView* rope, float eps,
                                float* workspace, unsigned* status, int num_sms,
                                cudaStream_t stream, void* state_out) {
    const int BH = B * H;
    cudaError_t e = configure(current_device());
    if (e != cudaSuccess) return e;
    uint8_t* state = state_out ? static_cast<uint8_t*>(state_out)
                               : reinterpret_cast<uint8_t*>(workspace) +
                                     tc_state_workspace_bytes(BH, N, num_sms);
    if ((e = launch_state(k, v, BH, N, rope, workspace, state, status, num_sms, stream)) !=
        cudaSuccess)
        return e;
    return launch_apply(q, g, state, out, BH, N, rope, eps, status, num_sms, kPdlState, stream);
}

}  // namespace sla
