// cla_internal.cuh -- shared host and device plumbing of libcla.so:
// status reporting, the workspace header, and the release/acquire flag
// protocol used by every cross-block carry (decoupled look-back).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>
#include <initializer_list>

#include "../../include/cla.h"

namespace cla {

// ----------------------------------------------------------------- host side
// Records a one-line description for cla_last_error_message() and returns
// the status unchanged.
int fail(int status, const char *fmt, ...);
int check_launch(const char *what);  // cudaGetLastError -> CLA_OK / CLA_ERR_CUDA
void clear_error();
// Raises func's dynamic shared memory limit to `bytes` on the current device,
// once per device: `done` (one per kernel) keeps a bit per device ordinal.
int set_max_dynamic_smem(std::atomic<unsigned long long> &done, const void *func, int bytes);
// Asks for the largest shared-memory carveout for func (once per device, as above), for
// kernels whose resident blocks per SM are bounded by shared memory.
int set_smem_carveout_max(std::atomic<unsigned long long> &done, const void *func);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned16_or_null(const void *p) { return p == nullptr || aligned16(p); }
// The product of non-negative sizes is below `limit`, computed so that it
// cannot overflow (a zero factor makes it 0).
inline bool product_below(std::initializer_list<int64_t> xs, double limit) {
    double p = 1.0;
    for (int64_t x : xs) p *= (double)x;
    return p < limit;
}
// Every non-NULL pointer a multiple of n bytes (n a power of two): the element
// alignment the kernels' plain loads and stores rely on.
inline bool aligned_or_null(std::initializer_list<const void *> ps, uintptr_t n) {
    for (const void *p : ps)
        if (p != nullptr && (reinterpret_cast<uintptr_t>(p) & (n - 1)) != 0) return false;
    return true;
}

// Every workspace starts with this header.  It is cleared (with the flag
// arrays that follow it) by one cudaMemsetAsync at the start of each call.
struct WsHeader {
    unsigned int ticket[8];   // per-kernel atomic tickets: block order of start
    unsigned int error;       // nonzero: a bounded wait gave up
    unsigned int where;       // which wait gave up (debug aid)
    unsigned int pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr unsigned int kErrTimeout = 1u;
// An input outside what a kernel handles was met on the device (data the host
// cannot check without a synchronisation); the results are not valid.
constexpr unsigned int kErrRange = 2u;

// Bound on polls of one flag (each poll after the first few sleeps ~100 ns):
// about a second before a block gives up, far beyond any legitimate wait.
constexpr unsigned int kSpinLimit = 1u << 23;

// Longest sequence of the tensor-core paths: their tensor-map loads take 32-bit token
// coordinates, which also reach one chunk before the first token and one past the last.
constexpr long long kMaxTokens = (1ll << 31) - 512;

// ----------------------------------------------------------------- device side
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned int *p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Loads that must observe another block's stores made visible by a release
// on a flag we acquired: bypass L1 (data written by other SMs).
__device__ __forceinline__ float4 ld_cg4(const float4 *p) { return __ldcg(p); }
__device__ __forceinline__ float ld_cg(const float *p) { return __ldcg(p); }

// Polls *flag until it is nonzero, at most kSpinLimit times.  On giving up
// records kErrTimeout in the header and returns 0; callers then proceed
// with a neutral value so that no other block waits on them forever.
__device__ __forceinline__ unsigned int wait_flag(const unsigned int *flag, WsHeader *hdr,
                                                  unsigned int where) {
    for (unsigned int it = 0; it < kSpinLimit; ++it) {
        unsigned int v = ld_acquire(flag);
        if (v != 0u) return v;
        if (it >= 8) __nanosleep(100);
    }
    atomicOr(&hdr->error, kErrTimeout);
    atomicExch(&hdr->where, where);
    return 0u;
}

}  // namespace cla

#define CLA_CUDA_TRY(expr, what)                                                    \
    do {                                                                            \
        cudaError_t e_ = (expr);                                                    \
        if (e_ != cudaSuccess)                                                      \
            return ::cla::fail(CLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e_)); \
    } while (0)
