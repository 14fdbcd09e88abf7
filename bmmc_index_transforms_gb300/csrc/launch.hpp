// Launchers of the device kernels (defined in kernels.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

#include "../../include/bmmc.h"
#include "planner.hpp"

namespace bmmc {

// One pass of a plan on `stream` (copy, per-element or tiled kernel).
cudaError_t launch_pass(const PassPlan& P, const void* in, void* out, cudaStream_t stream);

// The tiled kernel with an explicit grid (0 = one resident wave).
cudaError_t launch_tiled(const PassPlan& P, const void* in, void* out, cudaStream_t stream,
                         int grid_override);

// Plain copy of `bytes` bytes.
cudaError_t launch_copy(const void* in, void* out, size_t bytes, cudaStream_t stream);

// Copy out (and with clear, reset) the bounds record of the kernels of
// kernels.cu / lmad.cu / lmad_transpose_1_2.cu / lmad_transpose_4_8_16.cu:
// kRecordWords values (see bounds.cuh); all zero in
// builds without BMMC_BOUNDS_CHECK.
cudaError_t bounds_record_kernels(unsigned long long out[6], bool clear);
cudaError_t bounds_record_lmad(unsigned long long out[6], bool clear);
cudaError_t bounds_record_lmad_transpose_1_2(unsigned long long out[6], bool clear);
cudaError_t bounds_record_lmad_transpose_4_8_16(unsigned long long out[6], bool clear);
cudaError_t bounds_record_lmad_block(unsigned long long out[6], bool clear);
#ifdef BMMC_BOUNDS_CHECK
// The checks' self-test on a caller's device buffer of 512 bytes.
cudaError_t bounds_selftest(void* buf, cudaStream_t stream);
#endif

// OK when the GPU can read and write through p (device, managed or pinned
// memory, or pageable host memory on a device with pageable access).
bmmc_status pointer_reachable(const void* p);

}  // namespace bmmc
