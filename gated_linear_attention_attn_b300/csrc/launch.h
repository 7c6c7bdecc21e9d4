// Internal launchers of the linear-attention library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/sla.h"
#include "common.cuh"

namespace sla {

// Argument checks of the forward entry points (api.cu); fills *rv when RoPE is on.
sla_status_t check_forward(const void* q, const void* k, const void* v, const void* g,
                           const void* out, int B, int H, int N, int d,
                           const float* rope, float eps, size_t elem, RopeView* rv);

// fp32 SIMT path (simt.cu).
int simt_chunks(int BH, int N, int num_sms);
size_t simt_workspace_bytes(int BH, int C);
cudaError_t launch_simt_f32(const float* q, const float* k, const float* v, const float* g,
                            float* out, int B, int H, int N, const RopeView* rope, float eps,
                            float* workspace, int C, unsigned* status, cudaStream_t stream);

// The fp32 SIMT state partials (S_c in [m][n] order, then z_c) of C chunks
// per head, as simt_state_kernel writes them (simt.cu).
cudaError_t launch_simt_state_partials(const float* k, const float* v, int B, int H, int N,
                                       const RopeView* rope, float* partial, int C,
                                       unsigned* status, cudaStream_t stream);

// Backward (backward.cu): dq, dk, dv, dg of L = sum(dout * o).  bf16: six
// launches of the tensor-core state and apply kernels (five when the heads'
// states are given: state, tc_state_bytes as launch_tc_state writes them),
// workspace backward_bf16_workspace_bytes(BH, N, num_sms).  fp32:
// three launches over C chunks per head, workspace backward_workspace_bytes(BH, C).
size_t backward_workspace_bytes(int BH, int C);
size_t backward_bf16_workspace_bytes(int BH, int N, int num_sms);
cudaError_t launch_backward_bf16(const void* q, const void* k, const void* v, const void* g,
                                 const void* dout, void* dq, void* dk, void* dv, void* dg, int B,
                                 int H, int N, const RopeView* rope, float eps, float* workspace,
                                 int num_sms, unsigned* status, cudaStream_t stream,
                                 const void* state = nullptr);
cudaError_t launch_backward_f32(const float* q, const float* k, const float* v, const float* g,
                                const float* dout, float* dq, float* dk, float* dv, float* dg,
                                int B, int H, int N, const RopeView* rope, float eps,
                                float* workspace, int C, unsigned* status, cudaStream_t stream);

// Gated-softmax anchor forward (anchor.cu), bf16, head dim 256: the RoPE
// pre-pass (rotated k into workspace, anchor_workspace_bytes of it) when rope
// is given, then one tcgen05 attention launch (which rotates q itself).
size_t anchor_workspace_bytes(int BH, int N, bool rope);
cudaError_t launch_anchor(const void* q, const void* k, const void* v, const void* g, void* out,
                          int B, int H, int N, const RopeView* rope, void* workspace,
                          unsigned* status, cudaStream_t stream);

// AttnRes aggregation (attnres.cu): x = sum_n softmax_n(w . rmsnorm(s_n)) s_n
// per token over M <= kAttnResMaxSources bf16 [T][C] summaries, C a multiple
// of 256 up to 4096; one launch.
constexpr int kAttnResMaxSources = 8;
cudaError_t launch_attnres(const void* const* sources, int M, long long T, int C, const float* w,
                           float eps, void* out, unsigned* status, cudaStream_t stream);

// bf16 path on tcgen05 (tc_forward.cu).  The whole forward needs
// tc_workspace_bytes of workspace (counters, partial states, the heads'
// states); the state phase alone needs tc_state_workspace_bytes and writes
// tc_state_bytes of state.
size_t tc_workspace_bytes(int BH, int N, int num_sms);
// Bytes at the start of a workspace that hold the state kernel's per-head
// counters, which must read as zero when a launch starts (two-launch plan,
// state phase, backward, block-causal form).
size_t tc_counter_bytes(int BH);
size_t tc_state_workspace_bytes(int BH, int N, int num_sms);
size_t tc_state_bytes(int BH);
// The forward runs either as one fused launch (one cluster of C CTAs per
// head, no workspace) or as the state and apply launches.
// tc_forward_cluster gives C for the shape on device `dev`, 0 for the two
// launches.  Either also writes the heads' states (tc_state_bytes, the layout
// launch_tc_state writes) to state_out when it is not null.
int tc_forward_cluster(int dev, int BH, int N, bool rope, int num_sms);
cudaError_t launch_tc_fused(const void* q, const void* k, const void* v, const void* g, void* out,
                            int B, int H, int N, int C, const RopeView* rope, float eps,
                            unsigned* status, cudaStream_t stream, void* state_out = nullptr);
cudaError_t launch_tc_two_phase(const void* q, const void* k, const void* v, const void* g,
                                void* out, int B, int H, int N, const RopeView* rope, float eps,
                                float* workspace, unsigned* status, int num_sms,
                                cudaStream_t stream, void* state_out = nullptr);
// Block-causal form (tc_forward.cu): N = nb * block_tokens tokens per head,
// the RoPE rows of tokens [rope_offset, rope_offset + N) of the grid, carried
// states in and out (null for none).  Workspace: tc_workspace_bytes(B*H*nb,
// block_tokens, num_sms).
cudaError_t launch_tc_block_causal(const void* q, const void* k, const void* v, const void* g,
                                   void* out, int B, int H, int N, int block_tokens,
                                   const RopeView* rope, int rope_offset, float eps,
                                   const float* state_in, float* state_out, float* workspace,
                                   unsigned* status, int num_sms, cudaStream_t stream);
cudaError_t launch_tc_state(const void* k, const void* v, void* state, int B, int H, int N,
                            const RopeView* rope, void* workspace, unsigned* status, int num_sms,
                            cudaStream_t stream);
// mode: 0 the gated apply; 1 out = (R phi(q))^T S; 2 the backward's gate terms:
// with num = (R phi(q))^T S, den = phi(q) . z + eps and s = sigmoid(g), out = a =
// dout s / den, dg = dout num s (1 - s) / den and dden = -(a . num) / den per row
// ([B*H][N] fp32), and the partials of dS = sum (R phi(q)) a^T; 3 the masked gradient: out = [g > 0] (R^T (S q) + w z) with q
// as it is, g the tensor whose feature map is differentiated, z the state's, w =
// dden per row (1 when dden is null) and R the token's rotation (none without a
// table).
constexpr int kApplyGate = 0, kApplyRaw = 1, kApplyTerms = 2, kApplyGrad = 3;
// dspart (mode 2): the dS partial slots, tc_apply_partial_bytes; dzpart (mode 3,
// nullable): the dz partials sum_i dden_i phi(g_i), tc_apply_zpart_bytes.
// pdl: kPdlNone a plain launch; kPdlState a programmatic dependent of a kernel
// of ours that writes only the state (tiles are prefetched, the state waited
// for); kPdlWaitAll a programmatic dependent that waits before any read;
// kPdlWaitAllButG the same, except that the G tiles are inputs of the call,
// which the G producer prefetches without waiting.
constexpr int kPdlNone = 0, kPdlState = 1, kPdlWaitAll = 2, kPdlWaitAllButG = 3;
cudaError_t launch_tc_apply(const void* q, const void* g, const void* state, void* out, int B,
                            int H, int N, const RopeView* rope, float eps, unsigned* status,
                            int num_sms, cudaStream_t stream, int mode = kApplyGate,
                            const void* dout = nullptr, void* dg = nullptr,
                            float* dden = nullptr, float* dspart = nullptr,
                            float* dzpart = nullptr, int pdl = kPdlNone);
size_t tc_apply_partial_bytes(int BH, int N, int num_sms);
size_t tc_apply_zpart_bytes(int BH, int N, int num_sms);
// The dS state (bf16 S^T rows and fp32 z, as the state kernel writes a state)
// from the gate terms' dS partials and the masked gradient's dz partials.
// (pdl: launched as a programmatic dependent of the kernel before it)
cudaError_t launch_tc_ds_merge(const float* dspart, const float* dzpart, void* state, int B, int H,
                               int N, int num_sms, cudaStream_t stream, bool pdl = false);

// RoPE table (rope_table.cu): the header, then every token's pairs as fp16
// and as fp32, from the grid and band split or from caller-given fp32 pairs.
cudaError_t launch_rope_fill(float* table, int T, int Hs, int Ws, int dt, int dh, int dw,
                             float base, cudaStream_t stream);
cudaError_t launch_rope_from_pairs(float* table, const float* pairs, int N, int d,
                                   cudaStream_t stream);

// A one-thread kernel that waits on an mbarrier nobody arrives at and gives up
// after limit_ns, as every wait of the library's kernels does (selftest.cu).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned* status,
                                 cudaStream_t stream);

}  // namespace sla
