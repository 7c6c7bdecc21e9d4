// C ABI of the linear-attention library: argument checks, the per-stream
// workspace, and dispatch to the kernels.  Every check runs before anything
// is launched, so a call that returns an error has launched nothing.
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/sla.h"
#include "context.h"
#include "launch.h"

namespace sla {
namespace {

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    unsigned* status = nullptr;   // device status word (kStatusTimeout, ...)
};

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    size_t clean = 0;   // bytes at the start known to be zero when the stream's next launch runs
};

std::mutex g_mutex;
std::map<int, DeviceState> g_devices;
std::map<std::pair<int, uintptr_t>, Workspace> g_workspaces;

// Per-device set-up: SM count and the status word.  Called with g_mutex held.
sla_status_t device_state(int dev, DeviceState** out) {
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess)
            return SLA_ERR_CUDA;
        if (cudaMalloc(&st.status, 256) != cudaSuccess) return SLA_ERR_CUDA;
        if (cudaMemset(st.status, 0, 256) != cudaSuccess) return SLA_ERR_CUDA;
        st.ready = true;
    }
    *out = &st;
    return SLA_OK;
}

// The workspace of (dev, stream), grown to at least `bytes`.  Calls on one
// stream are ordered, so they can share it; calls on different streams get
// different workspaces.  Growing frees the old buffer (cudaFree waits for the
// device).  The first `counters` bytes hold per-head counters that must read
// zero when the launch starts: a completed launch leaves its counters at zero
// and writes its data after them, so the start of the buffer is cleared (on
// the stream, before the launch) only when a call's counters reach past what
// the previous call left zero, that is when the shape or the plan changes.
// Called with g_mutex held.
sla_status_t workspace(int dev, cudaStream_t stream, size_t bytes, void** out,
                       size_t counters = 0) {
    Workspace& ws = g_workspaces[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (ws.bytes < bytes) {
        if (ws.ptr) {
            cudaFree(ws.ptr);
            ws.ptr = nullptr;
            ws.bytes = 0;
        }
        const size_t rounded = (bytes + (1u << 20) - 1) & ~size_t((1u << 20) - 1);
        if (cudaMalloc(&ws.ptr, rounded) != cudaSuccess) {
            cudaGetLastError();
            return SLA_ERR_CUDA;
        }
        // the kernels' per-head counters must not start with a stale tag
        if (cudaMemsetAsync(ws.ptr, 0, rounded, stream) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(ws.ptr);
            ws.ptr = nullptr;
            return SLA_ERR_CUDA;
        }
        ws.bytes = rounded;
        ws.clean = rounded;
    }
    if (counters > ws.clean && cudaMemsetAsync(ws.ptr, 0, counters, stream) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    ws.clean = counters;
    *out = ws.ptr;
    return SLA_OK;
}

bool misaligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

}  // namespace

// Sizes: B, H, N >= 1 and d == 128, with B*H*N rows indexable by 32-bit ints.
static sla_status_t check_dims(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return SLA_ERR_INVALID_ARG;
    if (d != kHeadDim) return SLA_ERR_UNSUPPORTED;
    if ((long long)B * H * N > 0x7fffffffLL) return SLA_ERR_UNSUPPORTED;
    return SLA_OK;
}

static bool bad_eps(float eps) { return !std::isfinite(eps) || eps < 0.f; }

// A RoPE table pointer: NULL (no RoPE), else 256-byte aligned; the launch
// reads tokens [offset, offset + N) (exactly N tokens when exact).  What the
// table holds is checked on the device against its header (rope_table_ok);
// fills *rv.
static sla_status_t check_rope_range(const float* table, int N, int d, long long offset,
                                     bool exact, RopeView* rv) {
    if (!table) return SLA_OK;
    if (offset < 0) return SLA_ERR_INVALID_ARG;
    const long long need = offset + N;
    if (need > 0x7fffffffLL || (long long)rope_total_words(need, d) > 0x7fffffffLL)
        return SLA_ERR_UNSUPPORTED;
    if (misaligned(table, 256)) return SLA_ERR_ALIGNMENT;
    rv->hdr = reinterpret_cast<const uint32_t*>(table);
    rv->tok = rv->hdr + kRopeHeaderWords;
    rv->need = (int)need;
    rv->exact = exact ? 1 : 0;
    rv->d = d;
    return SLA_OK;
}

static sla_status_t check_rope(const float* table, int N, int d, RopeView* rv) {
    return check_rope_range(table, N, d, 0, true, rv);
}

// Buffers: none null, all 16-byte aligned, the output overlapping no input.
static sla_status_t check_buffers(const void* const* ins, const size_t* in_bytes, int n_ins,
                                  const void* out, size_t out_bytes) {
    for (int i = 0; i < n_ins; ++i)
        if (!ins[i]) return SLA_ERR_INVALID_ARG;
    if (!out) return SLA_ERR_INVALID_ARG;
    for (int i = 0; i < n_ins; ++i)
        if (misaligned(ins[i], 16)) return SLA_ERR_ALIGNMENT;
    if (misaligned(out, 16)) return SLA_ERR_ALIGNMENT;
    for (int i = 0; i < n_ins; ++i) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(out), y = reinterpret_cast<uintptr_t>(ins[i]);
        if (x < y + in_bytes[i] && y < x + out_bytes) return SLA_ERR_INVALID_ARG;
    }
    return SLA_OK;
}

// Checks shared by every forward entry point.  `elem` is the element size in
// bytes.
sla_status_t check_forward(const void* q, const void* k, const void* v, const void* g,
                           const void* out, int B, int H, int N, int d,
                           const float* rope, float eps, size_t elem, RopeView* rv) {
    if (!q || !k || !v || !g || !out) return SLA_ERR_INVALID_ARG;
    sla_status_t st = check_dims(B, H, N, d);
    if (st == SLA_ERR_INVALID_ARG) return st;
    if (bad_eps(eps)) return SLA_ERR_INVALID_ARG;
    if (st != SLA_OK) return st;
    const size_t bytes = (size_t)B * H * N * d * elem;
    const void* ins[4] = {q, k, v, g};
    const size_t sizes[4] = {bytes, bytes, bytes, bytes};
    if ((st = check_buffers(ins, sizes, 4, out, bytes)) != SLA_OK) return st;
    return check_rope(rope, N, d, rv);
}

}  // namespace sla

using namespace sla;

extern "C" {

size_t sla_rope_table_floats(int N, int d) {
    if (N < 1 || d < 2 || (d & 1)) return 0;
    const size_t words = rope_total_words(N, d);
    return words > 0x7fffffffULL ? 0 : words;
}

sla_status_t sla_rope_table_fill(float* table, int T, int Hs, int Ws, int d, int dt, int dh,
                                 int dw, float base, sla_stream_t stream) {
    if (!table) return SLA_ERR_INVALID_ARG;
    if (T < 1 || Hs < 1 || Ws < 1 || dt < 0 || dh < 0 || dw < 0) return SLA_ERR_INVALID_ARG;
    if ((dt | dh | dw) & 1 || dt + dh + dw != d || d < 2) return SLA_ERR_INVALID_ARG;
    if (!std::isfinite(base) || base <= 0.f) return SLA_ERR_INVALID_ARG;
    const long long N = (long long)T * Hs * Ws;
    if (N > 0x7fffffffLL || rope_total_words(N, d) > 0x7fffffffULL) return SLA_ERR_UNSUPPORTED;
    if (misaligned(table, 256)) return SLA_ERR_ALIGNMENT;
    if (launch_rope_fill(table, T, Hs, Ws, dt, dh, dw, base, (cudaStream_t)stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_rope_table_from_pairs(float* table, const float* pairs, int N, int d,
                                       sla_stream_t stream) {
    if (!table || !pairs || N < 1 || d < 2 || (d & 1)) return SLA_ERR_INVALID_ARG;
    if (rope_total_words(N, d) > 0x7fffffffULL) return SLA_ERR_UNSUPPORTED;
    if (misaligned(table, 256) || misaligned(pairs, 8)) return SLA_ERR_ALIGNMENT;
    const uintptr_t x = reinterpret_cast<uintptr_t>(table), y = reinterpret_cast<uintptr_t>(pairs);
    const size_t tbytes = rope_total_words(N, d) * 4, pbytes = (size_t)N * d * 4;
    if (x < y + pbytes && y < x + tbytes) return SLA_ERR_INVALID_ARG;
    if (launch_rope_from_pairs(table, pairs, N, d, (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

// Shared body of the forward entry points; state_out (bf16 only) receives the
// heads' states when not null.
static sla_status_t forward(const void* q, const void* k, const void* v, const void* g,
                            void* out, int B, int H, int N, int d,
                            const float* rope, float eps, sla_stream_t stream,
                            bool is_f32, void* state_out = nullptr) {
    RopeView rv{};
    sla_status_t st = check_forward(q, k, v, g, out, B, H, N, d, rope, eps,
                                    is_f32 ? sizeof(float) : 2, &rv);
    if (st != SLA_OK) return st;
    if (state_out) {                       // a further output: overlaps no other buffer
        const size_t bytes = (size_t)B * H * N * d * 2;
        const void* ins[5] = {q, k, v, g, out};
        const size_t sizes[5] = {bytes, bytes, bytes, bytes, bytes};
        if ((st = check_buffers(ins, sizes, 5, state_out, tc_state_bytes(B * H))) != SLA_OK)
            return st;
    }
    const RopeView* rp = rope ? &rv : nullptr;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    const int BH = B * H;
    void* ws = nullptr;
    cudaError_t err;
    if (is_f32) {
        const int C = simt_chunks(BH, N, ds->num_sms);
        if ((st = workspace(dev, s, simt_workspace_bytes(BH, C), &ws)) != SLA_OK) return st;
        err = launch_simt_f32((const float*)q, (const float*)k, (const float*)v,
                              (const float*)g, (float*)out, B, H, N, rp, eps, (float*)ws, C,
                              ds->status, s);
    } else if (const int C = tc_forward_cluster(dev, BH, N, rp != nullptr, ds->num_sms)) {
        err = launch_tc_fused(q, k, v, g, out, B, H, N, C, rp, eps, ds->status, s, state_out);
    } else {
        if ((st = workspace(dev, s, tc_workspace_bytes(BH, N, ds->num_sms), &ws,
                            tc_counter_bytes(BH))) != SLA_OK)
            return st;
        err = launch_tc_two_phase(q, k, v, g, out, B, H, N, rp, eps, (float*)ws, ds->status,
                                  ds->num_sms, s, state_out);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_linattn_forward(const void* q, const void* k, const void* v, const void* g,
                                 void* out, int B, int H, int N, int d,
                                 const float* rope_table, float eps,
                                 sla_stream_t stream) {
    return forward(q, k, v, g, out, B, H, N, d, rope_table, eps, stream, false);
}

sla_status_t sla_linattn_forward_f32(const float* q, const float* k, const float* v,
                                     const float* g, float* out, int B, int H, int N, int d,
                                     const float* rope_table, float eps,
                                     sla_stream_t stream) {
    return forward(q, k, v, g, out, B, H, N, d, rope_table, eps, stream, true);
}

sla_status_t sla_linattn_forward_keep_state(const void* q, const void* k, const void* v,
                                            const void* g, void* out, int B, int H, int N, int d,
                                            const float* rope_table, float eps, void* state,
                                            sla_stream_t stream) {
    if (!state) return SLA_ERR_INVALID_ARG;
    return forward(q, k, v, g, out, B, H, N, d, rope_table, eps, stream, false, state);
}

// Shared body of the backward entry points; `state` (bf16 only) is the heads'
// states of the forward, or null to recompute them.
static sla_status_t backward(const void* q, const void* k, const void* v, const void* g,
                             const void* dout, void* dq, void* dk, void* dv, void* dg, int B,
                             int H, int N, int d, const float* rope, float eps,
                             sla_stream_t stream, bool is_f32, const void* state = nullptr) {
    if (!q || !k || !v || !g || !dout || !dq || !dk || !dv || !dg) return SLA_ERR_INVALID_ARG;
    sla_status_t st = check_dims(B, H, N, d);
    if (st == SLA_ERR_INVALID_ARG) return st;
    if (bad_eps(eps)) return SLA_ERR_INVALID_ARG;
    if (st != SLA_OK) return st;
    const size_t bytes = (size_t)B * H * N * d * (is_f32 ? 4 : 2);
    const void* ins[6] = {q, k, v, g, dout, state};
    const size_t sizes[6] = {bytes, bytes, bytes, bytes, bytes, tc_state_bytes(B * H)};
    const int n_ins = state ? 6 : 5;
    void* outs[4] = {dq, dk, dv, dg};
    for (int i = 0; i < 4; ++i)
        if ((st = check_buffers(ins, sizes, n_ins, outs[i], bytes)) != SLA_OK) return st;
    for (int i = 0; i < 4; ++i)                      // the gradients overlap one another neither
        for (int j = i + 1; j < 4; ++j) {
            const uintptr_t x = reinterpret_cast<uintptr_t>(outs[i]);
            const uintptr_t y = reinterpret_cast<uintptr_t>(outs[j]);
            if (x < y + bytes && y < x + bytes) return SLA_ERR_INVALID_ARG;
        }
    RopeView rv{};
    if ((st = check_rope(rope, N, d, &rv)) != SLA_OK) return st;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    // fp32: one CTA per SM (a CTA holds S and S^T): chunks for whole waves of
    // two CTAs per SM at most, at least four 32-token tiles each
    const int tiles = (N + 31) / 32;
    int C = 2 * ds->num_sms / (B * H);
    if (C > (tiles + 3) / 4) C = (tiles + 3) / 4;
    if (C < 1) C = 1;
    void* ws = nullptr;
    const size_t ws_bytes = is_f32 ? backward_workspace_bytes(B * H, C)
                                   : backward_bf16_workspace_bytes(B * H, N, ds->num_sms);
    if ((st = workspace(dev, s, ws_bytes, &ws, is_f32 ? 0 : tc_counter_bytes(B * H))) != SLA_OK)
        return st;
    const RopeView* rp = rope ? &rv : nullptr;
    const cudaError_t err =
        is_f32 ? launch_backward_f32((const float*)q, (const float*)k, (const float*)v,
                                     (const float*)g, (const float*)dout, (float*)dq, (float*)dk,
                                     (float*)dv, (float*)dg, B, H, N, rp, eps, (float*)ws, C,
                                     ds->status, s)
               : launch_backward_bf16(q, k, v, g, dout, dq, dk, dv, dg, B, H, N, rp, eps,
                                      (float*)ws, ds->num_sms, ds->status, s, state);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_linattn_backward(const void* q, const void* k, const void* v, const void* g,
                                  const void* dout, void* dq, void* dk, void* dv, void* dg,
                                  int B, int H, int N, int d,
                                  const float* rope_table, float eps,
                                  sla_stream_t stream) {
    return backward(q, k, v, g, dout, dq, dk, dv, dg, B, H, N, d, rope_table, eps, stream, false);
}

sla_status_t sla_linattn_backward_f32(const float* q, const float* k, const float* v,
                                      const float* g, const float* dout, float* dq, float* dk,
                                      float* dv, float* dg, int B, int H, int N, int d,
                                      const float* rope_table, float eps,
                                      sla_stream_t stream) {
    return backward(q, k, v, g, dout, dq, dk, dv, dg, B, H, N, d, rope_table, eps, stream, true);
}

sla_status_t sla_linattn_backward_from_state(const void* q, const void* k, const void* v,
                                             const void* g, const void* dout, const void* state,
                                             void* dq, void* dk, void* dv, void* dg, int B, int H,
                                             int N, int d, const float* rope_table, float eps,
                                             sla_stream_t stream) {
    if (!state) return SLA_ERR_INVALID_ARG;
    return backward(q, k, v, g, dout, dq, dk, dv, dg, B, H, N, d, rope_table, eps, stream, false,
                    state);
}

sla_status_t sla_anchor_forward(const void* q, const void* k, const void* v, const void* g,
                                void* out, int B, int H, int N, int d,
                                const float* rope_table, sla_stream_t stream) {
    if (!q || !k || !v || !g || !out) return SLA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return SLA_ERR_INVALID_ARG;
    if (d != 256) return SLA_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535 || (long long)B * H * N > 0x7fffffffLL)
        return SLA_ERR_UNSUPPORTED;
    const size_t bytes = (size_t)B * H * N * d * 2;
    const void* ins[4] = {q, k, v, g};
    const size_t sizes[4] = {bytes, bytes, bytes, bytes};
    sla_status_t st = check_buffers(ins, sizes, 4, out, bytes);
    if (st != SLA_OK) return st;
    RopeView rv{};
    if ((st = check_rope(rope_table, N, d, &rv)) != SLA_OK) return st;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    void* ws = nullptr;
    if (rope_table &&
        (st = workspace(dev, s, anchor_workspace_bytes(B * H, N, true), &ws)) != SLA_OK)
        return st;
    if (launch_anchor(q, k, v, g, out, B, H, N, rope_table ? &rv : nullptr, ws, ds->status, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_attnres_aggregate(const void* const* sources, int M, int T, int C,
                                   const float* w, float eps, void* out, sla_stream_t stream) {
    if (!sources || !w || !out) return SLA_ERR_INVALID_ARG;
    if (M < 1 || T < 1 || C < 1 || bad_eps(eps)) return SLA_ERR_INVALID_ARG;
    if (M > kAttnResMaxSources || C % 256 != 0 || C > 4096) return SLA_ERR_UNSUPPORTED;
    const size_t bytes = (size_t)T * C * 2;
    for (int n = 0; n < M; ++n) {
        if (!sources[n]) return SLA_ERR_INVALID_ARG;
        if (misaligned(sources[n], 16)) return SLA_ERR_ALIGNMENT;
        const uintptr_t x = reinterpret_cast<uintptr_t>(out);
        const uintptr_t y = reinterpret_cast<uintptr_t>(sources[n]);
        if (x < y + bytes && y < x + bytes) return SLA_ERR_INVALID_ARG;
    }
    if (misaligned(out, 16) || misaligned(w, 16)) return SLA_ERR_ALIGNMENT;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    DeviceState* ds = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        sla_status_t st = device_state(dev, &ds);
        if (st != SLA_OK) return st;
    }
    if (launch_attnres(sources, M, T, C, w, eps, out, ds->status,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

size_t sla_linattn_carried_state_bytes(int B, int H, int d) {
    if (B < 1 || H < 1 || d != kHeadDim) return 0;
    return (size_t)B * H * (kHeadDim * kHeadDim + kHeadDim) * sizeof(float);
}

sla_status_t sla_linattn_forward_block_causal(const void* q, const void* k, const void* v,
                                              const void* g, void* out, int B, int H, int N,
                                              int d, int block_tokens,
                                              const float* rope_table,
                                              int rope_offset, float eps, const float* state_in,
                                              float* state_out, sla_stream_t stream) {
    if (!q || !k || !v || !g || !out) return SLA_ERR_INVALID_ARG;
    sla_status_t st = check_dims(B, H, N, d);
    if (st == SLA_ERR_INVALID_ARG) return st;
    if (bad_eps(eps)) return SLA_ERR_INVALID_ARG;
    if (st != SLA_OK) return st;
    if (block_tokens < 1 || N % block_tokens != 0) return SLA_ERR_INVALID_ARG;
    const size_t bytes = (size_t)B * H * N * d * 2;
    const size_t sbytes = sla_linattn_carried_state_bytes(B, H, d);
    const void* ins[4] = {q, k, v, g};
    const size_t sizes[4] = {bytes, bytes, bytes, bytes};
    if ((st = check_buffers(ins, sizes, 4, out, bytes)) != SLA_OK) return st;
    if (state_in && misaligned(state_in, 16)) return SLA_ERR_ALIGNMENT;
    if (state_out) {
        // the outgoing state overlaps no tensor and no incoming state but itself
        if (misaligned(state_out, 16)) return SLA_ERR_ALIGNMENT;
        const void* others[6] = {q, k, v, g, out, state_in};
        const size_t osizes[6] = {bytes, bytes, bytes, bytes, bytes, sbytes};
        for (int i = 0; i < 6; ++i) {
            if (!others[i] || (i == 5 && others[i] == state_out)) continue;
            const uintptr_t x = reinterpret_cast<uintptr_t>(state_out);
            const uintptr_t y = reinterpret_cast<uintptr_t>(others[i]);
            if (x < y + osizes[i] && y < x + sbytes) return SLA_ERR_INVALID_ARG;
        }
    }
    if (state_in) {
        // out is written while the incoming state may still be read
        const uintptr_t x = reinterpret_cast<uintptr_t>(state_in);
        const uintptr_t y = reinterpret_cast<uintptr_t>(out);
        if (x < y + bytes && y < x + sbytes) return SLA_ERR_INVALID_ARG;
    }
    RopeView rv{};
    if ((st = check_rope_range(rope_table, N, d, rope_offset, false, &rv)) != SLA_OK) return st;
    if (!rope_table && rope_offset != 0) return SLA_ERR_INVALID_ARG;
    const int nb = N / block_tokens;
    if ((long long)B * H * nb > 0x7fffffffLL / 2) return SLA_ERR_UNSUPPORTED;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    void* ws = nullptr;
    if ((st = workspace(dev, s, tc_workspace_bytes(B * H * nb, block_tokens, ds->num_sms), &ws,
                        tc_counter_bytes(B * H * nb))) != SLA_OK)
        return st;
    if (launch_tc_block_causal(q, k, v, g, out, B, H, N, block_tokens,
                               rope_table ? &rv : nullptr, rope_offset, eps, state_in, state_out,
                               (float*)ws, ds->status, ds->num_sms, s) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

int sla_linattn_forward_cluster(int B, int H, int N, int d, int rope) {
    if (check_dims(B, H, N, d) != SLA_OK) return -1;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if (device_state(dev, &ds) != SLA_OK) return -1;
    return tc_forward_cluster(dev, B * H, N, rope != 0, ds->num_sms);
}

size_t sla_linattn_state_bytes(int B, int H, int d) {
    if (B < 1 || H < 1 || d != kHeadDim) return 0;
    return tc_state_bytes(B * H);
}

sla_status_t sla_linattn_state(const void* k, const void* v, void* state, int B, int H, int N,
                               int d, const float* rope_table, sla_stream_t stream) {
    sla_status_t st = check_dims(B, H, N, d);
    if (st != SLA_OK) return st;
    const size_t bytes = (size_t)B * H * N * d * 2;
    const void* ins[2] = {k, v};
    const size_t sizes[2] = {bytes, bytes};
    if ((st = check_buffers(ins, sizes, 2, state, tc_state_bytes(B * H))) != SLA_OK) return st;
    RopeView rv{};
    if ((st = check_rope(rope_table, N, d, &rv)) != SLA_OK) return st;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    void* ws = nullptr;
    if ((st = workspace(dev, s, tc_state_workspace_bytes(B * H, N, ds->num_sms), &ws,
                        tc_counter_bytes(B * H))) != SLA_OK)
        return st;
    if (launch_tc_state(k, v, state, B, H, N, rope_table ? &rv : nullptr, ws, ds->status,
                        ds->num_sms, s) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_linattn_apply(const void* q, const void* g, const void* state, void* out, int B,
                               int H, int N, int d, const float* rope_table, float eps,
                               sla_stream_t stream) {
    sla_status_t st = check_dims(B, H, N, d);
    if (st == SLA_ERR_INVALID_ARG) return st;
    if (bad_eps(eps)) return SLA_ERR_INVALID_ARG;
    if (st != SLA_OK) return st;
    const size_t bytes = (size_t)B * H * N * d * 2;
    const void* ins[3] = {q, g, state};
    const size_t sizes[3] = {bytes, bytes, tc_state_bytes(B * H)};
    if ((st = check_buffers(ins, sizes, 3, out, bytes)) != SLA_OK) return st;
    RopeView rv{};
    if ((st = check_rope(rope_table, N, d, &rv)) != SLA_OK) return st;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    if ((st = device_state(dev, &ds)) != SLA_OK) return st;
    if (launch_tc_apply(q, g, state, out, B, H, N, rope_table ? &rv : nullptr, eps, ds->status,
                        ds->num_sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

sla_status_t sla_selftest_wait_timeout(unsigned int limit_us, sla_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000u) return SLA_ERR_INVALID_ARG;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    DeviceState* ds = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        sla_status_t st = device_state(dev, &ds);
        if (st != SLA_OK) return st;
    }
    if (launch_wait_selftest(1000ull * limit_us, ds->status,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}

const char* sla_status_string(sla_status_t status) {
    switch (status) {
        case SLA_OK: return "ok";
        case SLA_ERR_INVALID_ARG: return "invalid argument";
        case SLA_ERR_UNSUPPORTED: return "unsupported shape";
        case SLA_ERR_ALIGNMENT: return "misaligned pointer";
        case SLA_ERR_CUDA: return "CUDA runtime error";
        case SLA_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

sla_status_t sla_last_device_status(sla_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) return SLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* ds = nullptr;
    sla_status_t st = device_state(dev, &ds);
    if (st != SLA_OK) return st;
    unsigned word = 0;
    if (cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SLA_ERR_CUDA;
    if (word != 0 && cudaMemset(ds->status, 0, sizeof(word)) != cudaSuccess)
        return SLA_ERR_CUDA;
    if (word & kStatusTimeout) return SLA_ERR_DEVICE_TIMEOUT;
    if (word & kStatusBadTable) return SLA_ERR_INVALID_ARG;
    return word ? SLA_ERR_CUDA : SLA_OK;
}

}  // extern "C"
