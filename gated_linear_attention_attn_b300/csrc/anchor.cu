// Forward of the gated-softmax anchor layer on the tensor cores (bf16 in and
// out, fp32 accumulation).
//
// For one head (q, k, v, g: N x D with D = 256), with qr_i = R_i q_i and
// kr_j = R_j k_j (3D RoPE, or the identity):
//
//     o_i = sigmoid(g_i) * sum_j softmax_j(qr_i . kr_j / sqrt(D)) v_j
//
// "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section "Architecture")
// places these dense softmax layers at one layer in four, with 10 heads of 256
// (5B) or 16 heads of 256 (14B) and the Wan 3D rotary embedding; the arXiv
// abstract of 2607.21553 calls them gated-softmax anchors.
//
// Plan.  With RoPE, anchor_rope_kernel first writes the rotated k (bf16) to
// workspace.  anchor_attn_kernel then gives each CTA one tile of 128 queries
// of one head and streams that head's keys and values in tiles of 128:
//
//   warp 0      TMA producer: K in 64-dimension column blocks (16 KB) into a
//               ring of six, V in 64-key halves (32 KB) into a ring of two, in
//               the order the MMAs consume them (K two tiles ahead of V); K
//               and V are kept in L2 for the head's other CTAs;
//   warp 1      MMA issuer: S_j = Q K_j^T (M 128, N 128, K 256) into one of two
//               TMEM buffers, and O += P_j V_j (M 128, N 256, K 128) into a
//               256-column TMEM accumulator, in the order S_0, S_1, PV_0, S_2,
//               PV_1, ... so that S_{j+1} runs while P_j is formed;
//   warps 2-5   one query row per thread: first the row of q, rotated, into
//               shared memory; then per tile the row's 128 scores from TMEM,
//               the running maximum and sum, and P_j = 2^(s log2(e) / 16 - m)
//               in bf16 back into the S buffer (the PV product reads it from
//               TMEM); at the end o = sigmoid(g) O / l.
//
// Every MMA has N >= 128: the tensor core issues about one MMA per 64 cycles,
// so an M 128 x N 64 x K 16 product (32 cycles of math) would run at half rate.
//
// The running maximum m is only raised when a tile's maximum exceeds it by
// more than 2^8 (so P stays below 256, exact enough in bf16 and far from
// overflow); O and l are then rescaled in TMEM, after the PV product in
// flight has landed.  Keys past N are masked to zero weight; query rows past
// N are zero rows and not stored.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "launch.h"
#include "tc_ptx.cuh"

namespace sla {
namespace {

using namespace ptx;

constexpr int kAnD = 256;                             // head dim
constexpr int kAnM = 128;                             // queries per CTA
constexpr int kAnKeys = 128;                          // keys per tile
constexpr int kAnRowBytes = kAnD * 2;                 // one bf16 row: 512 B
constexpr int kAnQBox = kAnM * 128;                   // 64 columns of the Q tile: 16 KB
constexpr int kAnKChunk = kAnKeys * 128;              // 64 columns of a K tile: 16 KB
constexpr int kAnVBox = 64 * 128;                     // 64 keys x 64 columns of V: 8 KB
constexpr int kAnVHalf = 4 * kAnVBox;                 // 64 keys of a V tile: 32 KB
constexpr int kAnKSlots = 6;
constexpr int kAnVSlots = 2;
constexpr int kAnOffK = 4 * kAnQBox;                  // Q: 64 KB
constexpr int kAnOffV = kAnOffK + kAnKSlots * kAnKChunk;
constexpr int kAnOffBar = kAnOffV + kAnVSlots * kAnVHalf;   // 224 KB
constexpr int kAnBars = 1 + 2 * kAnKSlots + 2 * kAnVSlots + 4 + 3;
constexpr size_t kAnSmem = kAnOffBar + kAnBars * 8 + 16;
constexpr int kAnThreads = 192;
constexpr uint32_t kAnTmemCols = 512;
constexpr uint32_t kAnTmemO = 256;                    // O: columns [256, 512); S: 0 and 128
constexpr float kAnRescale = 8.f;                     // raise m only by more than 2^8
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kAnSmem <= 232448, "shared memory of one CTA");

struct AnchorParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* g;
    __nv_bfloat16* out;
    int N;
    int n_tiles;          // key tiles: ceil(N / 64)
    float scale_log2;     // log2(e) / sqrt(D)
    int rope;             // rotate q rows by `rv`
    RopeView rv;
    unsigned* status;
};

__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }

__global__ void __launch_bounds__(kAnThreads, 1)
anchor_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   AnchorParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAnOffBar);
    uint64_t* q_full = bars;                      // Q in shared memory (128 arrivals)
    uint64_t* k_full = bars + 1;                  // [kAnKSlots]
    uint64_t* k_empty = k_full + kAnKSlots;       // [kAnKSlots] the column block was read
    uint64_t* v_full = k_empty + kAnKSlots;       // [kAnVSlots]
    uint64_t* v_empty = v_full + kAnVSlots;       // [kAnVSlots] the half tile was read
    uint64_t* s_full = v_empty + kAnVSlots;       // [2] S_j in TMEM
    uint64_t* p_full = s_full + 2;                // [2] P_j in TMEM (128 arrivals)
    uint64_t* o_done = p_full + 2;                // one phase per PV product but the last
    uint64_t* o_final = o_done + 1;               // the last PV product
    uint64_t* mma_done = o_final + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kAnBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * kAnM;
    const int head = blockIdx.y;
    const int T = p.n_tiles;
    const uint32_t smem0 = smem_u32(smem);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 128);
        for (int s = 0; s < kAnKSlots; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kAnVSlots; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 128);
        }
        mbar_init(o_done, 1);
        mbar_init(o_final, 1);
        mbar_init(mma_done, 1);
        *abort_flag = (smem0 & 1023u) ? 1 : 0;    // the swizzled tiles need 1 KB alignment
        if (smem0 & 1023u) raise_status(p.status, kStatusLayout);
        if (p.rope && !rope_table_ok(p.rv)) {      // nothing of the table is read
            *abort_flag = 1;
            raise_status(p.status, kStatusBadTable);
        }
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kAnTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !*abort_flag) {
            const uint64_t keep = policy_evict_last();
            int kc = 0, vh = 0;                   // K column blocks and V halves issued
            bool ok = true;
            auto load_k = [&](int j) -> bool {    // the four column blocks of K_j
                for (int cb = 0; cb < 4; ++cb, ++kc) {
                    const int s = kc % kAnKSlots;
                    if (kc >= kAnKSlots &&
                        !mbar_wait(&k_empty[s], ((uint32_t)(kc / kAnKSlots) & 1u) ^ 1u, abort_flag,
                                   p.status))
                        return false;
                    mbar_arrive_expect_tx(&k_full[s], kAnKChunk);
                    tma_load_3d(smem + kAnOffK + s * kAnKChunk, &tm_k, &k_full[s], 64 * cb,
                                j * kAnKeys, head, keep);
                }
                return true;
            };
            auto load_v = [&](int j) -> bool {    // the two 64-key halves of V_j
                for (int h = 0; h < 2; ++h, ++vh) {
                    const int s = vh % kAnVSlots;
                    if (vh >= kAnVSlots &&
                        !mbar_wait(&v_empty[s], ((uint32_t)(vh / kAnVSlots) & 1u) ^ 1u, abort_flag,
                                   p.status))
                        return false;
                    mbar_arrive_expect_tx(&v_full[s], kAnVHalf);
                    for (int b = 0; b < 4; ++b)
                        tma_load_3d(smem + kAnOffV + s * kAnVHalf + b * kAnVBox, &tm_v, &v_full[s],
                                    64 * b, j * kAnKeys + 64 * h, head, keep);
                }
                return true;
            };
            // the MMAs' order: S_0, S_1, PV_0, S_2, PV_1, ...
            ok = load_k(0) && (T < 2 || load_k(1));
            for (int j = 0; ok && j < T; ++j) {
                ok = load_v(j);
                if (ok && j + 2 < T) ok = load_k(j + 2);
            }
            if (*abort_flag) {
                // copies still in flight land before the CTA exits
                for (int c = kc > kAnKSlots ? kc - kAnKSlots : 0; c < kc; ++c)
                    mbar_wait_drain(&k_full[c % kAnKSlots], (uint32_t)(c / kAnKSlots) & 1u);
                for (int c = vh > kAnVSlots ? vh - kAnVSlots : 0; c < vh; ++c)
                    mbar_wait_drain(&v_full[c % kAnVSlots], (uint32_t)(c / kAnVSlots) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kAnM, kAnKeys, false, false);
            constexpr uint32_t idesc_o = idesc_bf16(kAnM, kAnD, false, true);
            int kc = 0, vh = 0;
            // S_j = Q K_j^T: both K-major, 128-byte swizzled 64-column boxes
            // (16 dims = 32 bytes a step); each K column block is released
            // once its four MMAs are done.
            auto issue_s = [&](int j) -> bool {
                const uint32_t sb = tmem + (uint32_t)((j & 1) * kAnKeys);
                for (int cb = 0; cb < 4; ++cb, ++kc) {
                    const int s = kc % kAnKSlots;
                    if (!mbar_wait(&k_full[s], (uint32_t)(kc / kAnKSlots) & 1u, abort_flag, p.status))
                        return false;
                    tc_fence_after();
                    const uint32_t kb = smem0 + kAnOffK + s * kAnKChunk;
                    const uint32_t qb = smem0 + cb * kAnQBox;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(sb, smem_desc_sw128(qb + ks * 32, 16, 1024),
                                 smem_desc_sw128(kb + ks * 32, 16, 1024), idesc_s,
                                 (cb > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&k_empty[s]);
                }
                mma_commit(&s_full[j & 1]);
                return true;
            };
            // O += P_j V_j: P from TMEM (the first 64 columns of S_j's buffer,
            // 16 keys = 8 columns a step); V MN-major per 64-key half (16 keys
            // = 2048 bytes a step, the four 64-column boxes kAnVBox apart).
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(&p_full[j & 1], (uint32_t)(j >> 1) & 1u, abort_flag, p.status))
                    return false;
                tc_fence_after();
                const uint32_t pb = tmem + (uint32_t)((j & 1) * kAnKeys);
                for (int h = 0; h < 2; ++h, ++vh) {
                    const int s = vh % kAnVSlots;
                    if (!mbar_wait(&v_full[s], (uint32_t)(vh / kAnVSlots) & 1u, abort_flag, p.status))
                        return false;
                    tc_fence_after();
                    const uint32_t vb = smem0 + kAnOffV + s * kAnVHalf;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts(tmem + kAnTmemO, pb + (uint32_t)((h * 4 + ks) * 8),
                                    smem_desc_sw128(vb + ks * 2048, kAnVBox, 1024), idesc_o,
                                    (j > 0 || h > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&v_empty[s]);
                }
                mma_commit(j == T - 1 ? o_final : o_done);
                return true;
            };
            bool ok = !*abort_flag && mbar_wait(q_full, 0, abort_flag, p.status);
            if (ok) tc_fence_after();
            for (int j = 0; ok && j < T; ++j) {
                ok = issue_s(j);
                if (ok && j > 0) ok = issue_pv(j - 1);
            }
            if (ok) issue_pv(T - 1);
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0);
        }
    } else {
        // ------------------------------------------------ Q, softmax and epilogue
        const int quad = warp & 3;                 // TMEM lanes 32 quad .. 32 quad + 31
        const int r = quad * 32 + lane;            // this thread's query row in the tile
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        const int row = q0 + r;
        const bool live = row < p.N;
        const size_t base = ((size_t)head * p.N + (size_t)(live ? row : 0)) * kAnD;
        bool ok = !*abort_flag;
        {   // this row of q (rotated, or zero past N) into the swizzled Q tile:
            // column block cb at cb * 16 KB, 16-byte chunk c of row r at
            // position c xor (r mod 8) of the row's 128 bytes
            const uint4* q4 = reinterpret_cast<const uint4*>(p.q + base);
            // this token's (cos, sin) pairs; the table is read only when it checked out
            const float2* cs = p.rope && ok ? rope_pairs(p.rv) + (size_t)(live ? row : 0) * (kAnD / 2)
                                            : nullptr;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 u = live ? ldg_nc_na128(q4 + cb * 8 + c) : make_uint4(0, 0, 0, 0);
                    if (cs) {
                        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float2 f = bf2_to_f2(w[i]);
                            rotate_pair(f.x, f.y, __ldg(cs + cb * 32 + c * 4 + i));
                            w[i] = f2_to_bf2(f.x, f.y);
                        }
                        u = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    sts128(smem0 + cb * kAnQBox + r * 128 + ((uint32_t)(c ^ (r & 7)) << 4), u);
                }
            }
            fence_proxy_async_smem();                // Q visible to the tensor core
            mbar_arrive(q_full);
        }
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; ok && j < T; ++j) {
            const int s = j & 1;
            ok = warp_all(mbar_wait(&s_full[s], (uint32_t)(j >> 1) & 1u, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sb = trow + (uint32_t)(s * kAnKeys);
            float x[128];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t xa[32];
                tmem_ld32(sb + (uint32_t)(32 * q), xa);
#pragma unroll
                for (int c = 0; c < 32; ++c) x[32 * q + c] = __uint_as_float(xa[c]);
            }
            tmem_ld_wait();
            const int valid = p.N - j * kAnKeys;     // keys of this tile inside the head
            if (valid < kAnKeys) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= valid) x[c] = -INFINITY;
            }
            float mx8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx8[c] = fmaxf(x[c], x[c + 8]);
#pragma unroll
            for (int c = 16; c < 128; c += 8)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], x[c + i]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_tile = mx * p.scale_log2;
            const bool grow = m_tile > m_used + kAnRescale;
            if (!warp_all(!grow)) {                  // some row of the warp raises m
                const float m_new = grow ? m_tile : m_used;
                const float f = ex2_approx(m_used - m_new);   // 0 on the first tile
                l *= f;
                if (j > 0) {
                    // O holds PV_0 .. PV_{j-2}; PV_{j-1} may still be running
                    ok = warp_all(mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, p.status));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kAnD; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(trow + kAnTmemO + (uint32_t)c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                        tmem_st32(trow + kAnTmemO + (uint32_t)c, o);
                    }
                    tmem_st_wait();
                }
                m_used = m_new;
            }
            // P row: 128 keys in bf16 pairs over the buffer's first 64 columns
            const float2 sc = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm = make_float2(-m_used, -m_used);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pw[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = 64 * h + 2 * i;
                    const float2 t = fma2(make_float2(x[c], x[c + 1]), sc, nm);
                    const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
                    acc[i & 3] = fma2(e, make_float2(1.f, 1.f), acc[i & 3]);
                    pw[i] = f2_to_bf2(e.x, e.y);
                }
                tmem_st32(sb + (uint32_t)(32 * h), pw);
            }
            l += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                 ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
            tmem_st_wait();
            tc_fence_before();                       // P_j in TMEM before the MMA reads it
            mbar_arrive(&p_full[s]);
        }
        if (ok) ok = warp_all(mbar_wait(o_final, 0, abort_flag, p.status));
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            const uint4* g4 = reinterpret_cast<const uint4*>(p.g + base);
            uint4* o4 = reinterpret_cast<uint4*>(p.out + base);
#pragma unroll 1
            for (int c = 0; c < kAnD; c += 32) {
                uint32_t o[32];
                tmem_ld32(trow + kAnTmemO + (uint32_t)c, o);
                uint4 gv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    gv[i] = live ? ldg_nc_na128(g4 + c / 8 + i) : make_uint4(0, 0, 0, 0);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
                        uint32_t ow[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 gg = bf2_to_f2(gw[t]);
                            const float s0 = rcp_approx(1.f + ex2_approx(-gg.x * kLog2e));
                            const float s1 = rcp_approx(1.f + ex2_approx(-gg.y * kLog2e));
                            ow[t] = f2_to_bf2(__uint_as_float(o[8 * i + 2 * t]) * inv_l * s0,
                                              __uint_as_float(o[8 * i + 2 * t + 1]) * inv_l * s1);
                        }
                        o4[c / 8 + i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kAnTmemCols);
    }
}

// kr = R k per token row (bf16 in and out), 32 threads a row, eight
// dimensions (four pairs) each; the angles from the table's fp32 pairs.
__global__ void __launch_bounds__(256)
anchor_rope_kernel(const uint4* __restrict__ k, uint4* __restrict__ kr, int N, long long rows,
                   RopeView rope, unsigned* status) {
    const long long row = (long long)blockIdx.x * 8 + threadIdx.x / 32;
    const int c = threadIdx.x % 32;
    if (!rope_table_ok(rope)) {               // nothing of the table is read
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(status, kStatusBadTable);
        return;
    }
    if (row >= rows) return;
    const float2* cs = rope_pairs(rope) + (size_t)(row % N) * (kAnD / 2);
    const size_t at = (size_t)row * (kAnD / 8) + c;
    const uint4 u = __ldg(k + at);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = bf2_to_f2(w[i]);
        rotate_pair(f.x, f.y, __ldg(cs + 4 * c + i));
        o[i] = f2_to_bf2(f.x, f.y);
    }
    kr[at] = make_uint4(o[0], o[1], o[2], o[3]);
}

PFN_cuTensorMapEncodeTiled_v12000 anchor_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// A [BH][N][256] bf16 tensor as 3D (d fastest), boxes of 64 columns x `rows`
// tokens x 1 head, 128-byte swizzle; rows past N read as zero.
bool anchor_map(CUtensorMap* m, const void* base, int N, int BH, int rows) {
    auto fn = anchor_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kAnD, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kAnRowBytes, (cuuint64_t)N * kAnRowBytes};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t anchor_workspace_bytes(int BH, int N, bool rope) {
    return rope ? (size_t)BH * N * kAnRowBytes : 0;
}

cudaError_t launch_anchor(const void* q, const void* k, const void* v, const void* g, void* out,
                          int B, int H, int N, const RopeView* rope, void* workspace,
                          unsigned* status, cudaStream_t stream) {
    const int BH = B * H;
    const void* ka = k;
    if (rope) {
        uint4* kr = static_cast<uint4*>(workspace);
        const long long rows = (long long)BH * N;
        anchor_rope_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>((const uint4*)k, kr, N,
                                                                           rows, *rope, status);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ka = kr;
    }
    CUtensorMap mk, mv;
    if (!anchor_map(&mk, ka, N, BH, kAnKeys) || !anchor_map(&mv, v, N, BH, 64))
        return cudaErrorInvalidValue;
    {   // the shared-memory opt-in, once per device
        static std::mutex mu;
        static bool done[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!done[dev]) {
            e = cudaFuncSetAttribute(anchor_attn_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAnSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    AnchorParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.g = static_cast<const __nv_bfloat16*>(g);
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.N = N;
    prm.n_tiles = (N + kAnKeys - 1) / kAnKeys;
    prm.scale_log2 = kLog2e / 16.f;                 // log2(e) / sqrt(256)
    prm.rope = rope ? 1 : 0;
    prm.rv = rope ? *rope : RopeView{};
    prm.status = status;
    const dim3 grid((unsigned)((N + kAnM - 1) / kAnM), (unsigned)BH);
    anchor_attn_kernel<<<grid, kAnThreads, kAnSmem, stream>>>(mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace sla
