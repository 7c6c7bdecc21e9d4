// Host side of the entry points: the device a call runs on.
#pragma once

#include <cuda_runtime.h>

namespace sla {

// The calling thread's current device, with that device's primary context made
// current in the thread.  The tensor maps are encoded through the driver API,
// which needs a current context; a thread that has only ever asked for its
// device (a framework's worker thread, say) has none yet, and the encoding
// then fails with an invalid-context error.
inline cudaError_t bind_current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    return e == cudaSuccess ? cudaSetDevice(*dev) : e;
}

}  // namespace sla
