// Optional device-side bounds checks for every kernel of the library.
//
// A build compiled with -DBMMC_BOUNDS_CHECK makes each global and shared
// memory access of the kernels test its address first:
//   - a global load must lie inside the launch's source buffer, a global
//     store inside its destination buffer (the [lo, hi) byte ranges the
//     launcher passes as one extra kernel argument);
//   - a load of a whole aligned word that may hold bytes next to the copied
//     elements (the 16-byte chunks and 4-byte words some LMAD kernels fetch)
//     must start on a multiple of its size and overlap the source buffer:
//     such a word lies in the page of a byte of the buffer;
//   - a shared-memory access must lie inside one of the shared arrays the
//     kernel registered on entry.
// An access that fails is skipped (a load yields zero), and the failure is
// counted in a device record of this translation unit: the number of
// failures and, for the first one, the site (file tag * 100000 + source
// line), the address, the range it was tested against and the access size.
// The host reads and clears the record through bmmc_bounds_report.  Nothing
// traps or waits: a failing access only leaves wrong bytes behind.
//
// Without BMMC_BOUNDS_CHECK every test below is the constant true and the
// extra kernel argument does not exist, so the kernels compile to the same
// code as without this header.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace bmmc {
namespace chk {

struct Span {
    uintptr_t lo, hi;  // [lo, hi) in bytes
};

// The buffers one launch may touch: the source and the destination.
struct Bounds {
    Span in, out;
};

__host__ __device__ inline Bounds bounds(const void* in, uint64_t in_bytes, const void* out, uint64_t out_bytes) {
    return Bounds{{(uintptr_t)in, (uintptr_t)in + in_bytes}, {(uintptr_t)out, (uintptr_t)out + out_bytes}};
}

// Slots of the device record.
enum { kFailures = 0, kSite, kAddress, kLo, kHi, kBytes, kRecordWords };

#ifdef BMMC_BOUNDS_CHECK

constexpr bool kEnabled = true;

// One record per translation unit (each .cu file is compiled on its own).
static __device__ unsigned long long g_record[kRecordWords];

// The launch's buffers and up to three shared arrays, written by every
// thread on entry (all with the same values, each thread reading back its
// own write, so no barrier is needed).
struct Entry {
    Bounds b;
    uint32_t sh_lo[3], sh_hi[3];
};
static __shared__ Entry s_entry;

static __device__ __noinline__ void fail(int site, uintptr_t addr, uintptr_t lo, uintptr_t hi, unsigned bytes) {
    const unsigned long long k = atomicAdd(&g_record[kFailures], 1ull);
    if (k == 0) {
        g_record[kSite] = (unsigned long long)site;
        g_record[kAddress] = addr;
        g_record[kLo] = lo;
        g_record[kHi] = hi;
        g_record[kBytes] = bytes;
    }
}

__device__ __forceinline__ uint32_t sh_off(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void enter(const Bounds& b, const void* s0 = nullptr, uint32_t n0 = 0,
                                      const void* s1 = nullptr, uint32_t n1 = 0, const void* s2 = nullptr,
                                      uint32_t n2 = 0) {
    s_entry.b = b;
    const void* s[3] = {s0, s1, s2};
    const uint32_t n[3] = {n0, n1, n2};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        s_entry.sh_lo[i] = s[i] ? sh_off(s[i]) : 0u;
        s_entry.sh_hi[i] = s[i] ? sh_off(s[i]) + n[i] : 0u;
    }
}

__device__ __forceinline__ bool inside(const void* p, unsigned bytes, const Span& s, int site) {
    const uintptr_t a = (uintptr_t)p;
    if (a >= s.lo && a <= s.hi && bytes <= s.hi - a) return true;
    fail(site, a, s.lo, s.hi, bytes);
    return false;
}

__device__ __forceinline__ bool in_ok(const void* p, unsigned bytes, int site) {
    return inside(p, bytes, s_entry.b.in, site);
}
__device__ __forceinline__ bool out_ok(const void* p, unsigned bytes, int site) {
    return inside(p, bytes, s_entry.b.out, site);
}
// A whole aligned word of `bytes` (a power of two) that must hold at least
// one byte of the source buffer.
__device__ __forceinline__ bool in_word_ok(const void* p, unsigned bytes, int site) {
    const uintptr_t a = (uintptr_t)p;
    const Span& s = s_entry.b.in;
    if ((a & (bytes - 1)) == 0 && a < s.hi && a + bytes > s.lo) return true;
    fail(site, a, s.lo, s.hi, bytes);
    return false;
}
__device__ __forceinline__ bool sh_ok(const void* p, unsigned bytes, int site) {
    const uint32_t a = sh_off(p);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (a >= s_entry.sh_lo[i] && a + bytes <= s_entry.sh_hi[i] && a + bytes >= a) return true;
    fail(site, a, s_entry.sh_lo[0], s_entry.sh_hi[0], bytes);
    return false;
}

// Host: copy this translation unit's record out and optionally clear it.
static inline cudaError_t read_record(unsigned long long out[kRecordWords], bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_record, sizeof(unsigned long long) * kRecordWords);
    if (e == cudaSuccess && clear) {
        const unsigned long long zero[kRecordWords] = {};
        e = cudaMemcpyToSymbol(g_record, zero, sizeof(zero));
    }
    return e;
}

// Bytes of dynamic shared memory the block was launched with.
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

#define BMMC_CHK_PARAM , const ::bmmc::chk::Bounds bmmc_chk_bounds
#define BMMC_CHK_PTYPE , const ::bmmc::chk::Bounds
#define BMMC_CHK_ARG(b) , (b)
#define BMMC_CHK_ENTER(...) ::bmmc::chk::enter(bmmc_chk_bounds, __VA_ARGS__)
#define BMMC_CHK_ENTER_GLOBAL() ::bmmc::chk::enter(bmmc_chk_bounds)
#define BMMC_CHK_SITE (BMMC_CHK_FILE * 100000 + __LINE__)
#define BMMC_IN_OK(p, n) ::bmmc::chk::in_ok((p), (unsigned)(n), BMMC_CHK_SITE)
#define BMMC_IN_WORD_OK(p, n) ::bmmc::chk::in_word_ok((p), (unsigned)(n), BMMC_CHK_SITE)
#define BMMC_OUT_OK(p, n) ::bmmc::chk::out_ok((p), (unsigned)(n), BMMC_CHK_SITE)
#define BMMC_SH_OK(p, n) ::bmmc::chk::sh_ok((p), (unsigned)(n), BMMC_CHK_SITE)

#else  // !BMMC_BOUNDS_CHECK

constexpr bool kEnabled = false;

static inline cudaError_t read_record(unsigned long long out[kRecordWords], bool) {
    for (int i = 0; i < kRecordWords; ++i) out[i] = 0;
    return cudaSuccess;
}

#define BMMC_CHK_PARAM
#define BMMC_CHK_PTYPE
#define BMMC_CHK_ARG(b)
#define BMMC_CHK_ENTER(...) ((void)0)
#define BMMC_CHK_ENTER_GLOBAL() ((void)0)
#define BMMC_IN_OK(p, n) true
#define BMMC_IN_WORD_OK(p, n) true
#define BMMC_OUT_OK(p, n) true
#define BMMC_SH_OK(p, n) true

#endif  // BMMC_BOUNDS_CHECK

}  // namespace chk
}  // namespace bmmc
