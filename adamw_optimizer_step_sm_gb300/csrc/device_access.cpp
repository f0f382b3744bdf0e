// device_access.cpp -- checks, before any kernel runs, that every buffer of a
// tensor list can be dereferenced by the plan's device, so a wrong pointer is
// an error code rather than a GPU fault.
//
// Accepted: device memory of that device; managed memory; pinned host memory
// mapped at the same address (the kernels then read or write it over the
// CPU-GPU link, NVLink-C2C on Grace systems); and pageable host memory on
// devices that report pageable-memory access (address-translation services).
#include <cuda_runtime_api.h>

#include "adamw_internal.h"

namespace adamw {

int check_device_access(const adamw_tensor_t* table, int32_t n, int32_t mode, int device) {
    int64_t es[5];
    element_sizes(mode, es);
    int pageable = 0;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, device) != cudaSuccess) {
        set_cuda_error("cudaDeviceGetAttribute", cudaGetErrorString(cudaGetLastError()));
        return ADAMW_ERR_CUDA;
    }
    for (int32_t k = 0; k < n; ++k) {
        const adamw_tensor_t& t = table[k];
        if (t.numel == 0) continue;
        const void* ptrs[5] = {t.param, t.grad, t.exp_avg, t.exp_avg_sq, t.aux};
        for (int s = 0; s < 5; ++s) {
            if (es[s] == 0) continue;  // a buffer the mode does not use
            const void* p = ptrs[s];
            cudaPointerAttributes a{};
            if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
                set_cuda_error("cudaPointerGetAttributes", cudaGetErrorString(cudaGetLastError()));
                return ADAMW_ERR_NOT_ACCESSIBLE;
            }
            bool ok = false;
            switch (a.type) {
                case cudaMemoryTypeDevice: ok = (a.device == device); break;
                case cudaMemoryTypeManaged: ok = true; break;
                case cudaMemoryTypeHost: ok = (a.devicePointer == p); break;
                default: ok = (pageable != 0); break;  // unregistered host memory
            }
            if (!ok) return ADAMW_ERR_NOT_ACCESSIBLE;
        }
    }
    return ADAMW_OK;
}

}  // namespace adamw
