// bmmc_permute_static_scratch: the two-factor permute without any device
// allocation.  Its scratch is one file-scope device array; the host looks up
// that array's device address once per device (cudaGetSymbolAddress, with
// the device current) and hands it to the same launch path the other
// two-factor entry points use.  In host code the array's name only stands
// for a host-side shadow symbol, so its address is never passed to a kernel
// directly.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/bmmc.h"
#include "launch.hpp"
#include "planner.hpp"

static __device__ __align__(256) unsigned char g_bmmc_static_scratch[BMMC_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static array on the current device (looked up on
// the first call per device, then cached).
bmmc_status static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return BMMC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_bmmc_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return BMMC_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return BMMC_OK;
}

bool ranges_overlap(const void* a, const void* b, size_t bytes) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bytes && y < x + bytes;
}

// The buffers must be memory the GPU can reach: device, managed or pinned
// memory, or pageable memory on a device that can access it.
bmmc_status reachable(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    if (attr.type != cudaMemoryTypeUnregistered) return BMMC_OK;
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
        cudaGetLastError();
        return BMMC_ERR_CUDA;
    }
    return pageable ? BMMC_OK : BMMC_ERR_INVALID_ARG;
}

}  // namespace

extern "C" bmmc_status bmmc_permute_static_scratch(bmmc_plan_t plan, const void* in, void* out,
                                                   void* stream) {
    if (!plan || !in || !out) return BMMC_ERR_INVALID_ARG;
    if (plan->mode != BMMC_MODE_TWO_FACTOR) return BMMC_ERR_INVALID_ARG;
    const size_t bytes = ((size_t)1 << plan->n) * (size_t)plan->elem;
    if (bytes > BMMC_STATIC_SCRATCH_BYTES) return BMMC_ERR_TOO_LARGE;
    if (((uintptr_t)in | (uintptr_t)out) & 15u) return BMMC_ERR_MISALIGNED;
    if (ranges_overlap(in, out, bytes)) return BMMC_ERR_ALIAS;
    bmmc_status s = reachable(in);
    if (s == BMMC_OK) s = reachable(out);
    if (s != BMMC_OK) return s;
    void* scratch = nullptr;
    if ((s = static_scratch_address(&scratch)) != BMMC_OK) return s;
    if (ranges_overlap(scratch, in, bytes) || ranges_overlap(scratch, out, bytes)) return BMMC_ERR_ALIAS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bmmc::launch_pass(plan->first_pass, in, scratch, st) != cudaSuccess) return BMMC_ERR_CUDA;
    if (bmmc::launch_pass(plan->second_pass, scratch, out, st) != cudaSuccess) return BMMC_ERR_CUDA;
    return BMMC_OK;
}
