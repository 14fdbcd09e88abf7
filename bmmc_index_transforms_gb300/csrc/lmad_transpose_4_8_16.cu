// LMAD transposes of 4-, 8- and 16-byte words (the kernels are in
// lmad_transpose.cuh).
#include "../../include/bmmc.h"
#define BMMC_CHK_FILE 4  // site tag of this file in bounds-checked builds
#include "bounds.cuh"
#include "lmad_internal.hpp"
#include "lmad_transpose.cuh"

namespace bmmc {
namespace lmad {

cudaError_t launch_transpose_wide(const void* in, void* out, size_t word, const LmadCopy& C, cudaStream_t s) {
    switch (word) {
        case 4: return launch_transpose_w(static_cast<const Word<4>::T*>(in), static_cast<Word<4>::T*>(out), C, s);
        case 8: return launch_transpose_w(static_cast<const Word<8>::T*>(in), static_cast<Word<8>::T*>(out), C, s);
        case 16: return launch_transpose_w(static_cast<const Word<16>::T*>(in), static_cast<Word<16>::T*>(out), C, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lmad

// Read (and optionally clear) the bounds record of this file's kernels.
cudaError_t bounds_record_lmad_transpose_4_8_16(unsigned long long out[chk::kRecordWords], bool clear) {
    return chk::read_record(out, clear);
}

}  // namespace bmmc
