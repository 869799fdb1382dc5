// Host-side check that a caller's buffer is memory the library's kernels may
// use: device memory of the handle's device, or managed memory.  Host
// memory (pageable or pinned) is refused before any launch, so a wrong
// pointer becomes an argument error instead of a fault on the device.
#pragma once

#include <cstdio>

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

}  // namespace hk
