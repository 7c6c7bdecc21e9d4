// The allocation-free variant of the bf16 forward: the same tensor-core
// kernels as sla_linattn_forward, with their scratch memory (the split-N
// partial states) taken from a fixed array that is part of the library's
// device image instead of from cudaMalloc.
//
// The array is allocated by the CUDA runtime when the library's device code
// is loaded on a GPU and stays allocated on every GPU that loaded it until the
// process exits.  Host code cannot use the array's name as a device address:
// the address is looked up once per device with cudaGetSymbolAddress.
#include <mutex>

#include "context.h"
#include "launch.h"

namespace sla {
namespace {

constexpr size_t kScratchBytes = size_t(24) << 20;   // 24 MiB, shared by every call

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    int num_sms = 0;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
    size_t clean = kScratchBytes;       // bytes at its start known to be zero (all, at load)
};

std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_devices[kMaxDevices];

// One-time set-up of device `dev` (which is current): the SM count and the
// device address of the scratch array.  Called with g_noalloc_mutex held.
sla_status_t noalloc_device(int dev, NoAllocDevice** out) {
    if (dev < 0 || dev >= kMaxDevices) return SLA_ERR_UNSUPPORTED;
    NoAllocDevice& st = g_noalloc_devices[dev];
    if (!st.ready) {
        if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess) {
            cudaGetLastError();
            return SLA_ERR_CUDA;
        }
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return SLA_ERR_CUDA;
        }
        st.scratch = static_cast<unsigned char*>(ptr);
        st.ready = true;
    }
    *out = &st;
    return SLA_OK;
}

}  // namespace
}  // namespace sla

using namespace sla;

extern "C" sla_status_t sla_linattn_forward_noalloc(const void* q, const void* k, const void* v,
                                                    const void* g, void* out, int B, int H,
                                                    int N, int d,
                                                    const float* rope_table,
                                                    float eps, unsigned int* device_status,
                                                    sla_stream_t stream) {
    RopeView rv{};
    sla_status_t st = check_forward(q, k, v, g, out, B, H, N, d, rope_table, eps, 2, &rv);
    if (st != SLA_OK) return st;
    if (reinterpret_cast<uintptr_t>(device_status) % sizeof(unsigned) != 0)
        return SLA_ERR_ALIGNMENT;
    int dev = 0;
    if (bind_current_device(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice* nd = nullptr;
    if ((st = noalloc_device(dev, &nd)) != SLA_OK) return st;
    const int BH = B * H;
    const RopeView* rp = rope_table ? &rv : nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    const int C = tc_forward_cluster(dev, BH, N, rp != nullptr, nd->num_sms);
    // The per-head counters at the start of the array must read zero: a
    // completed call leaves its own at zero and its data after them, so the
    // start is cleared (a memset on the stream, no allocation) only when this
    // call's counters reach past what the previous call left zero.
    auto counters_clean = [&](size_t counters) -> bool {
        if (counters > nd->clean && cudaMemsetAsync(nd->scratch, 0, counters, s) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        nd->clean = counters;
        return true;
    };
    if (C != 0) {
        // the fused kernel needs no scratch
        err = launch_tc_fused(q, k, v, g, out, B, H, N, C, rp, eps, device_status, s);
    } else {
        // the whole scratch this shape needs must fit in the fixed array
        if (tc_workspace_bytes(BH, N, nd->num_sms) > kScratchBytes) return SLA_ERR_UNSUPPORTED;
        if (!counters_clean(tc_counter_bytes(BH))) return SLA_ERR_CUDA;
        err = launch_tc_two_phase(q, k, v, g, out, B, H, N, rp, eps,
                                  reinterpret_cast<float*>(nd->scratch), device_status,
                                  nd->num_sms, s);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SLA_ERR_CUDA;
    }
    return SLA_OK;
}
