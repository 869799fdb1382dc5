// Host-side helpers of the C ABI:
//   * the check that a caller's buffer is memory the library's kernels may
//     use (device memory of the handle's device, or managed memory); host
//     memory, pageable or pinned, is refused before any launch, so a wrong
//     pointer becomes an argument error instead of a fault on the device;
//   * binding a context on a thread before the library's driver calls.
#pragma once

#include <cstdio>

#include <cuda.h>
#include <cuda_runtime.h>

namespace hk {

// nullptr when `p` qualifies; otherwise the reason, written into buf.
inline const char* device_ptr_problem(const void* p, int dev, char (&buf)[128]) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // the query's error is not sticky; clear it
        std::snprintf(buf, sizeof(buf), "is not a pointer CUDA knows");
        return buf;
    }
    if (a.type == cudaMemoryTypeManaged) return nullptr;
    if (a.type != cudaMemoryTypeDevice) {
        std::snprintf(buf, sizeof(buf), "is host memory, not device memory");
        return buf;
    }
    if (a.device != dev) {
        std::snprintf(buf, sizeof(buf), "is on device %d, the handle on device %d", a.device, dev);
        return buf;
    }
    return nullptr;
}

// The driver calls the library makes (tensor-map encoding) need a context
// current on the calling thread, and a thread whose first CUDA call on the
// device is one of the library's may have none: runtime calls bind the
// device's primary context only when they themselves need it.  This binds
// the current device's primary context when no context is current, and
// leaves any current context alone.
inline cudaError_t ensure_context() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    static const GetCurrentFn get_current = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<GetCurrentFn>(p);
        return static_cast<GetCurrentFn>(nullptr);
    }();
    CUcontext c = nullptr;
    if (get_current && get_current(&c) == CUDA_SUCCESS && c != nullptr) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaSetDevice(dev);  // makes the device's primary context current
}

}  // namespace hk
