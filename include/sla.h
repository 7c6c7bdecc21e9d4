/*
 * sla.h -- C ABI of the gated bidirectional linear-attention forward
 * (SANA-Video 2.0), a single-GPU CUDA library for B300 (sm_103a), with the
 * layer's backward and block-causal form, the gated-softmax anchor layer and
 * the AttnRes aggregation (declared further down).
 *
 * The operation.  "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md,
 * section "Architecture") builds 75% of its attention layers as gated
 * bidirectional linear attention with Wan 3D rotary position embeddings, 20
 * heads x 128 in the 5B model and 32 x 128 in the 14B model; the arXiv
 * abstract of 2607.21553 calls it the gated linear attention used for the
 * O(N)-dominated token mixing.  For each (batch b, head h), with q, k, v, g
 * the N x d slices of that head:
 *
 *     phi(x) = max(x, 0)
 *     S      = sum_j R_j phi(k_j) v_j^T          (d x d; R_j = I without RoPE)
 *     z      = sum_j phi(k_j)                    (d, never rotated)
 *     o_i    = sigmoid(g_i) * (R_i phi(q_i))^T S / (phi(q_i) . z + eps)
 *
 * The sums run over all N tokens (bidirectional: no causal mask).  The gate
 * g has the shape of q and acts elementwise.  R_n is the 3D rotary embedding
 * of token n, applied to the numerator only (see the RoPE table below).
 *
 * Layout.  q, k, v, g and out are [B][H][N][d] row-major and contiguous
 * (d fastest), all in device memory of the current device.  out has the
 * element type of the inputs.
 *
 * Ownership.  The caller owns every buffer passed in.  The library owns a
 * workspace per (device, stream) for the split-N partial states and the
 * heads' states of the two-launch plan (about 66 KB per SM of the device plus
 * 99 KB per head; the fused plan needs none), and for the scratch of the
 * backward and of the anchor layer with RoPE (sizes at those entry points),
 * allocated with cudaMalloc on the first call that needs it (or more of it)
 * and kept until the process exits.  A call that has to grow the workspace
 * synchronises the device; make the first call of the largest shape outside
 * stream capture.  The start of a workspace holds per-head counters that
 * must read zero when a kernel starts; a call of another shape or plan on the
 * same stream may clear it first (cudaMemsetAsync on the stream), so a
 * captured graph expects no call of another shape on its stream between its
 * capture and its replays.
 *
 * Errors.  Every argument is checked before anything is launched; a call
 * that returns an error has launched nothing.  Calls are asynchronous on
 * `stream` (NULL = the legacy default stream); SLA_ERR_CUDA reports a launch
 * error.  Kernels never spin forever: a wait that exceeds its limit (about
 * one second) sets a device status word and the kernel returns early;
 * sla_last_device_status() reads (and clears) that word.
 */
#ifndef SLA_H_
#define SLA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle: the same type as cudaStream_t. */
typedef struct CUstream_st* sla_stream_t;

typedef enum sla_status {
    SLA_OK = 0,
    SLA_ERR_INVALID_ARG = 1,    /* null pointer, size < 1, bad eps, aliasing, bad RoPE table */
    SLA_ERR_UNSUPPORTED = 2,    /* a shape the kernels do not implement (e.g. d != 128) */
    SLA_ERR_ALIGNMENT = 3,      /* a tensor not 16-byte aligned (a RoPE table not 256-byte aligned) */
    SLA_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, allocation, no device) */
    SLA_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up a wait and returned early */
} sla_status_t;

/*
 * The 3D rotary embedding ("Wan 3D rotary position embeddings", NVlabs page,
 * "Architecture"; RoFormer's rotation).  Token n of a T x Hs x Ws latent grid
 * (one token per latent cell, "(1, 1, 1) latent patches") sits at
 * n = (t*Hs + h)*Ws + w.  The head dimension is split into three even bands
 * [0, dt), [dt, dt+dh), [dt+dh, d) that take t, h and w respectively; inside
 * a band of width W, pair j = (x_{2p}, x_{2p+1}) turns by pos * base^(-2j/W)
 * radians (complex multiplication of x_{2p} + i x_{2p+1}).
 *
 * The RoPE table argument of every entry point (`rope_table`) is NULL for no
 * rotation, or a device buffer of sla_rope_table_floats(N, d) 4-byte words,
 * 256-byte aligned, written by sla_rope_table_fill or
 * sla_rope_table_from_pairs.  With P = d/2 pairs per token it holds:
 *
 *   words [0, 64)               a header: word 0 the tag 0x33414c53, word 1
 *                               the layout version (1), word 2 the number of
 *                               tokens N, word 3 d, words 4-6 the grid
 *                               (T, Hs, Ws), words 7-9 the bands (dt, dh, dw),
 *                               word 10 the base as an fp32 bit pattern (grid,
 *                               bands and base are 0 for a table made from
 *                               pairs), word 11 the offset of the fp16 rows
 *                               (64), word 12 the offset of the fp32 pairs
 *                               (64 + N*P); the rest 0;
 *   words [64, 64 + N*P)        per token n, its P pairs as fp16 (cos, sin)
 *                               (cos in the low half of the word), read by the
 *                               tensor-core kernels next to the token's row;
 *   words [64 + N*P, 64 + 3N*P) per token n, its P pairs as fp32 (cos, sin):
 *                               the plain [N][d/2][2] table, read by the fp32
 *                               and anchor kernels.
 *
 * The host checks only the pointer (NULL or 256-byte aligned).  Every kernel
 * that rotates first checks the header: the tag, the version, d, and the
 * number of tokens (exactly the call's N, or at least rope_offset + N for the
 * block-causal form).  On a mismatch it reads nothing more of the table and
 * sets a bit of the device status word, which sla_last_device_status reports
 * as SLA_ERR_INVALID_ARG; the call's outputs are then undefined.  The buffer
 * must hold at least the 64 header words.
 */

/* 4-byte words of a RoPE table for N tokens of head dimension d (0 if invalid). */
size_t sla_rope_table_floats(int N, int d);

/*
 * Writes the RoPE table (layout above) of a T x Hs x Ws grid, N = T*Hs*Ws,
 * bands (dt, dh, dw) with dt + dh + dw == d, all even (44/42/42 for d = 128,
 * 88/84/84 for d = 256), base `base` (10000 for the Wan embedding), into
 * `table`.  The angles are formed and the cosine and sine taken in double
 * precision, rounded to fp32, and the fp32 values rounded to fp16.
 * Asynchronous on `stream`.
 */
sla_status_t sla_rope_table_fill(float* table, int T, int Hs, int Ws, int d, int dt, int dh,
                                 int dw, float base, sla_stream_t stream);

/*
 * Writes a RoPE table (layout above) from caller-given angles: `pairs` is a
 * device array [N][d/2][2] of fp32 (cos, sin), 8-byte aligned, not
 * overlapping `table`; it is copied into the fp32 part and rounded to fp16 for
 * the other.  For callers that already hold a plain per-token table.
 * Asynchronous on `stream`; `pairs` may be freed once the copy has run.
 */
sla_status_t sla_rope_table_from_pairs(float* table, const float* pairs, int N, int d,
                                       sla_stream_t stream);

/*
 * The forward with bf16 q, k, v, g and out (IEEE bfloat16, 2 bytes each),
 * fp32 accumulation.  B, H, N >= 1; d must be 128.  rope_table: NULL for no
 * RoPE, else a RoPE table (layout above) of exactly N tokens built for d.
 * eps: finite, >= 0 (1e-6 in the workloads).  All five tensors 16-byte
 * aligned; out must not overlap any input.  Asynchronous on `stream`.
 */
sla_status_t sla_linattn_forward(const void* q, const void* k, const void* v, const void* g,
                                 void* out, int B, int H, int N, int d,
                                 const float* rope_table, float eps,
                                 sla_stream_t stream);

/*
 * The same forward for fp32 tensors (fp32 arithmetic throughout, no tensor
 * cores), same arguments, layout and errors.
 */
sla_status_t sla_linattn_forward_f32(const float* q, const float* k, const float* v,
                                     const float* g, float* out, int B, int H, int N, int d,
                                     const float* rope_table, float eps,
                                     sla_stream_t stream);

/*
 * How sla_linattn_forward runs a shape on the current device.  The bf16
 * forward has two launch plans.  One fused launch gives every head a cluster
 * of C CTAs (2 <= C <= 8): each CTA sums its share of the head's keys and
 * values, the cluster adds the partial states through distributed shared
 * memory, and each CTA applies the state to its share of the queries.  This
 * needs no workspace.  It applies when every head's cluster can be resident
 * at once (B*H clusters of C CTAs on the device's SMs) and the head has at
 * least C tiles of 128 queries.  It is taken when it applies and either N is
 * at most 64 * 128 = 8192 tokens or its B*H*C CTAs cover at least 85% of the
 * SMs (otherwise the two launches measured faster on B300).  Otherwise the
 * forward launches the state kernel and then the apply kernel
 * (sla_linattn_state, sla_linattn_apply).
 *
 * Returns C for the fused launch, 0 for the two launches, -1 for an invalid
 * shape (rope: nonzero when a RoPE table will be passed).  The environment
 * variable SLA_FORWARD_KERNEL, read on every call, overrides the choice:
 * "split" always takes the two launches, "fused" the fused launch wherever it
 * applies (the same rule as without it).
 */
int sla_linattn_forward_cluster(int B, int H, int N, int d, int rope);

/*
 * The two phases of sla_linattn_forward, for callers that reuse a state
 * (several query sets against one set of keys and values) or time the phases.
 * When sla_linattn_forward_cluster returns 0, sla_linattn_forward is exactly
 * sla_linattn_state followed by sla_linattn_apply, except that it keeps the
 * state in the library's workspace and lets the apply kernel start while the
 * state kernel finishes (the fused launch sums the partial states in another
 * order, so its output may differ in the last bits).
 *
 * The state of one head is sla_linattn_state_bytes(1, 1, 128) = 33280 bytes:
 * S^T (row n = output dim, column m = key dim) as bf16 in the layout the
 * tensor cores read (two 64-column halves of 128 rows x 128 bytes; the
 * 16-byte chunk c of row n sits at chunk position (c mod 8) xor (n mod 8) of
 * its row), then z as 128 fp32 values.  Heads follow each other, b-major.
 */
size_t sla_linattn_state_bytes(int B, int H, int d);   /* 0 if the shape is invalid */

/*
 * Phase 1: S~ = sum_j R_j phi(k_j) v_j^T and z = sum_j phi(k_j) for every
 * head of bf16 k and v ([B][H][N][d], device).  state: device buffer of
 * sla_linattn_state_bytes(B, H, d) bytes, 16-byte aligned, overlapping
 * neither input.  rope_table as for sla_linattn_forward (N tokens of k).
 * Uses the library's per-stream workspace for the split-N partial states.
 */
sla_status_t sla_linattn_state(const void* k, const void* v, void* state, int B, int H, int N,
                               int d, const float* rope_table, sla_stream_t stream);

/*
 * Phase 2: out = sigmoid(g) * (R phi(q)) S~ / (phi(q) . z + eps) for bf16 q
 * and g ([B][H][N][d], device; N query tokens, which may differ from the N of
 * the state's keys), with a state written by sla_linattn_state for the same
 * B and H.  rope_table as for sla_linattn_forward, for the N query tokens.
 * out must overlap neither q, g nor the state.
 */
sla_status_t sla_linattn_apply(const void* q, const void* g, const void* state, void* out, int B,
                               int H, int N, int d, const float* rope_table, float eps,
                               sla_stream_t stream);

/*
 * Block-causal form with a carried state ("SANA-Video" model card, "Constant-
 * Memory KV Cache for Block Linear Attention": block-wise autoregressive
 * generation that keeps global context in the cumulative state of linear
 * attention at a fixed memory cost).  The N tokens of each head form N /
 * block_tokens consecutive blocks (whole latent frames, so block_tokens =
 * frames per block * Hs * Ws).  A token of block b attends to its own block in
 * both directions and to every earlier block through the running state:
 *
 *     S_b = S_in + sum_{j in blocks 0..b} R_j phi(k_j) v_j^T
 *     z_b = z_in + sum_{j in blocks 0..b} phi(k_j)
 *     o_i = sigmoid(g_i) * (R_i phi(q_i))^T S_b / (phi(q_i) . z_b + eps)
 *
 * and the outgoing state is (S_last, z_last).  With block_tokens = N and no
 * incoming state this is sla_linattn_forward.  Calls on consecutive
 * stretches of a sequence, each passing the previous call's state_out as its
 * state_in, give the same result as one call on the whole sequence.
 *
 * Arguments as for sla_linattn_forward (bf16 q, k, v, g, out), plus:
 * block_tokens: >= 1, dividing N.  rope_table: NULL or a table of at least
 * rope_offset + N tokens: this call's token n is token rope_offset + n of the
 * table (absolute positions, so a later stretch of a video passes its first
 * token's index); rope_offset must be 0 without RoPE.
 * state_in, state_out: NULL (a zero incoming state; no outgoing state) or
 * device buffers of sla_linattn_carried_state_bytes(B, H, d) bytes, 16-byte
 * aligned: per head (b-major) S as 128 x 128 fp32 row-major (row m = key
 * dim, column n = value dim), then z as 128 fp32.  The running sums are kept
 * in fp32; state_out may equal state_in (updated in place) but must not
 * overlap anything else, and state_in must not overlap out.  Uses the
 * library's per-stream workspace (about 66 KB per SM plus 99 KB per block of
 * every head).
 */
size_t sla_linattn_carried_state_bytes(int B, int H, int d);   /* 0 if the shape is invalid */
sla_status_t sla_linattn_forward_block_causal(const void* q, const void* k, const void* v,
                                              const void* g, void* out, int B, int H, int N,
                                              int d, int block_tokens,
                                              const float* rope_table,
                                              int rope_offset, float eps, const float* state_in,
                                              float* state_out, sla_stream_t stream);

/*
 * Backward of the layer: the gradients of L = sum(dout * o) for the o of
 * sla_linattn_forward (bf16, fp32 arithmetic) or sla_linattn_forward_f32
 * (fp32), as the models of "SANA-Video 2.0" (NVlabs/Sana
 * docs/sana_video2.md, section "Training") are trained through the layer.
 * With num_i = (R_i phi(q_i))^T S, den_i = phi(q_i) . z + eps,
 * s_i = sigmoid(g_i):
 *
 *     a_i    = dout_i * s_i / den_i,    dg_i = dout_i * num_i / den_i * s_i (1 - s_i)
 *     dden_i = -(a_i . num_i) / den_i
 *     dS = sum_i (R_i phi(q_i)) a_i^T,  dz = sum_i dden_i phi(q_i)
 *     dq_i = [q_i > 0] (R_i^T (S a_i) + dden_i z)
 *     dk_j = [k_j > 0] (R_j^T (dS v_j) + dz),   dv_j = dS^T R_j phi(k_j)
 *
 * (the ReLU derivative at 0 is 0).  q, k, v, g, dout: inputs as for the
 * forward; dq, dk, dv, dg: outputs of the same shape, layout and type, none
 * overlapping an input or another output.  rope_table and eps as for the
 * forward.  The state S, z is recomputed from k and v.  bf16: the six
 * contractions (S, num, dS, S a, dS v, dS^T kr) run on the tensor cores with
 * bf16 operands and fp32 accumulation, S and dS rounded to bf16, the
 * elementwise terms in fp32; the per-stream workspace holds the state
 * kernel's partials, the two states, two [B*H*N][128] bf16 scratch tensors
 * and B*H*N floats.  fp32: everything on the fp32 FMA units, with a
 * workspace of 2 * 66 KB per chunk of every head.
 */
sla_status_t sla_linattn_backward(const void* q, const void* k, const void* v, const void* g,
                                  const void* dout, void* dq, void* dk, void* dv, void* dg,
                                  int B, int H, int N, int d,
                                  const float* rope_table, float eps,
                                  sla_stream_t stream);
sla_status_t sla_linattn_backward_f32(const float* q, const float* k, const float* v,
                                      const float* g, const float* dout, float* dq, float* dk,
                                      float* dv, float* dg, int B, int H, int N, int d,
                                      const float* rope_table, float eps,
                                      sla_stream_t stream);

/*
 * Training without recomputing the state.  A training step runs the forward
 * and then the backward of the same q, k, v, g; the backward above sums S, z
 * over k and v again.  sla_linattn_forward_keep_state is sla_linattn_forward
 * (same launches, same output) that also writes each head's state, as
 * sla_linattn_state writes it (bf16 S^T, then z in fp32; the two-launch plan
 * gives the very bytes sla_linattn_state gives, the fused plan the sum of its
 * cluster's partials in rank order), into `state`: a device buffer of
 * sla_linattn_state_bytes(B, H, d) bytes, 16-byte aligned, overlapping no
 * other argument.  sla_linattn_backward_from_state is sla_linattn_backward
 * (bf16) with that state as S, z instead of its own: one launch and two
 * tensor passes (k and v) fewer.  Its gradients equal sla_linattn_backward's
 * bit for bit when the state is the one sla_linattn_state or the two-launch
 * plan gives for the same k and v; the state is only read, and no output may
 * overlap it.
 */
sla_status_t sla_linattn_forward_keep_state(const void* q, const void* k, const void* v,
                                            const void* g, void* out, int B, int H, int N, int d,
                                            const float* rope_table, float eps, void* state,
                                            sla_stream_t stream);
sla_status_t sla_linattn_backward_from_state(const void* q, const void* k, const void* v,
                                             const void* g, const void* dout, const void* state,
                                             void* dq, void* dk, void* dv, void* dg, int B, int H,
                                             int N, int d, const float* rope_table, float eps,
                                             sla_stream_t stream);

/*
 * Forward of the gated-softmax anchor layer ("SANA-Video 2.0", NVlabs/Sana
 * docs/sana_video2.md, section "Architecture": one attention layer in four is
 * a dense softmax layer, 10 heads of 256 in the 5B model, 16 in the 14B
 * model, with the Wan 3D rotary embedding; the arXiv abstract of 2607.21553
 * calls them gated-softmax anchors).  Per (batch, head), with
 * qr_i = R_i q_i and kr_j = R_j k_j (R the identity without RoPE):
 *
 *     o_i = sigmoid(g_i) * sum_j softmax_j(qr_i . kr_j / sqrt(d)) v_j
 *
 * over all N keys (no mask), the gate elementwise.  q, k, v, g, out: bf16
 * [B][H][N][d] row-major and contiguous in device memory, 16-byte aligned,
 * out overlapping no input; d must be 256 (SLA_ERR_UNSUPPORTED otherwise),
 * B * H <= 65535.  rope_table: NULL, or a RoPE table of exactly N tokens
 * built for d = 256 (the Wan split is 88/84/84).  Scores and
 * the output are accumulated in fp32 on the tensor cores; the rotated q and k
 * and the softmax weights enter the products rounded to bf16.  With RoPE the
 * rotated k goes to the library's per-stream workspace (B*H*N*d*2 bytes).
 * Asynchronous on `stream`.
 */
sla_status_t sla_anchor_forward(const void* q, const void* k, const void* v, const void* g,
                                void* out, int B, int H, int N, int d,
                                const float* rope_table, sla_stream_t stream);

/*
 * Block Attention Residual (AttnRes) aggregation ("SANA-Video 2.0",
 * NVlabs/Sana docs/sana_video2.md, section "Architecture": a shared,
 * timestep-independent Attention Residual aggregation in blocks of eight
 * layers; the arXiv abstract of 2607.21553: completed block summaries are
 * routed into later linear layers).  The pages give no formula; this entry
 * point computes the reading, per token t:
 *
 *     k_n(t) = s_n(t) / sqrt(mean_c s_n(t, c)^2 + eps)
 *     x(t)   = sum_n softmax_n(w . k_n(t)) s_n(t)
 *
 * sources: a HOST array of M device pointers, each a bf16 [T][C] row-major
 * summary (16-byte aligned); 1 <= M <= 8.  C must be a multiple of 256, at
 * most 4096 (SLA_ERR_UNSUPPORTED otherwise; 2560 and 4096 in the models).  w: device, C fp32 values (the shared
 * query, any RMS-norm gain folded in), 16-byte aligned.  out: device bf16
 * [T][C], overlapping no source.  eps finite, >= 0.  fp32 arithmetic.
 * Asynchronous on `stream`; the host array may be freed on return.
 */
sla_status_t sla_attnres_aggregate(const void* const* sources, int M, int T, int C,
                                   const float* w, float eps, void* out, sla_stream_t stream);

/*
 * The bf16 forward of sla_linattn_forward for callers that cannot allocate
 * device memory.  No page has a counterpart: this entry point exists for
 * library users, not for the method.  Some callers must not see a library
 * allocate: a framework whose caching allocator has already reserved the
 * device's memory (a cudaMalloc of ours could fail or fragment its pool), a
 * runtime whose enqueue path forbids allocation (plugin interfaces), or a
 * latency-critical loop that cannot afford the device-wide synchronisation of
 * cudaMalloc and cudaFree.  This call allocates nothing: it runs the same
 * kernels with their scratch (the split-N partial states) in a fixed 24 MiB
 * array that is part of the library's device code.  Each GPU that loads the
 * library holds that array until the process exits.
 *
 * Arguments, layout and checks are those of sla_linattn_forward, plus:
 * device_status: NULL, or a caller-owned device pointer to a 4-byte aligned
 * unsigned int into which the kernels OR a nonzero value when they return
 * early: 1 if one of their waits gave up, 4 if the RoPE table's header does
 * not fit the call (the word is never cleared by the library).  With NULL,
 * such an early return is not reported.
 *
 * Size limit: the fused launch (see sla_linattn_forward_cluster) needs no
 * scratch.  For the two launches, a shape whose scratch does not fit in the
 * 24 MiB array returns SLA_ERR_UNSUPPORTED before anything is launched.  That
 * scratch is about 66 KB x (number of SMs + B*H) + 33 KB x B*H, so B*H up to
 * about 150 heads fits on a 148-SM B300.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array, which keeps the
 * last call's contents.  The only values a call reads before writing them are
 * per-head counters at the start of the array, which must read zero: the state
 * kernel returns the counters it used to zero before it exits, and a call
 * whose counters reach past those the previous call left zero (a call with
 * more heads) first clears the start of the array with cudaMemsetAsync on
 * `stream` (no allocation).  The counters also carry a tag of the call that
 * set them, so a count left by a call that gave up a wait reads as zero to the
 * next call.  Calls that overlap on the GPU (other streams, other host
 * threads) race on the array; order them on one stream or with events.
 */
sla_status_t sla_linattn_forward_noalloc(const void* q, const void* k, const void* v,
                                         const void* g, void* out, int B, int H, int N, int d,
                                         const float* rope_table, float eps,
                                         unsigned int* device_status, sla_stream_t stream);

/*
 * Self-test of the kernels' bounded waits: launches one thread that waits on
 * an mbarrier nobody arrives at, with the same wait the library's kernels use,
 * and gives up after limit_us microseconds (1 .. 1000000), setting the device
 * status word as a kernel does when a wait runs out.  The next
 * sla_last_device_status(stream) then returns SLA_ERR_DEVICE_TIMEOUT (and
 * clears the word).  Nothing else runs and no memory but the status word is
 * touched, so the device stays usable.  Asynchronous on `stream`.
 */
sla_status_t sla_selftest_wait_timeout(unsigned int limit_us, sla_stream_t stream);

/* A static, human-readable name for a status code. */
const char* sla_status_string(sla_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: SLA_ERR_DEVICE_TIMEOUT if a kernel gave up a wait since the
 * last read, SLA_ERR_INVALID_ARG if a kernel found a RoPE table whose header
 * does not fit its call, SLA_ERR_CUDA if the synchronisation failed, else
 * SLA_OK.
 */
sla_status_t sla_last_device_status(sla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SLA_H_ */
