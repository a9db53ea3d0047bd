// api.cu -- status reporting shared by every entry point of libcla.so.
#include <stdarg.h>
#include <stdio.h>

#include "cla_internal.cuh"

namespace cla {

static thread_local char g_msg[512] = "";

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

void clear_error() { g_msg[0] = '\0'; }

int check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(CLA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return CLA_OK;
}

int set_max_dynamic_smem(std::atomic<unsigned long long> &done, const void *func, int bytes) {
    int dev = 0;
    CLA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    // ordinals beyond 63 are not cached: the attribute is then set on every call
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return CLA_OK;
    CLA_CUDA_TRY(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                 "cudaFuncSetAttribute");
    done.fetch_or(bit, std::memory_order_acq_rel);
    return CLA_OK;
}

int set_smem_carveout_max(std::atomic<unsigned long long> &done, const void *func) {
    int dev = 0;
    CLA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0ull && (done.load(std::memory_order_acquire) & bit) != 0ull) return CLA_OK;
    CLA_CUDA_TRY(cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, 100),
                 "cudaFuncSetAttribute");
    done.fetch_or(bit, std::memory_order_acq_rel);
    return CLA_OK;
}

}  // namespace cla

extern "C" const char *cla_status_string(int status) {
    switch (status) {
        case CLA_OK: return "CLA_OK";
        case CLA_ERR_INVALID_ARG: return "CLA_ERR_INVALID_ARG";
        case CLA_ERR_UNSUPPORTED: return "CLA_ERR_UNSUPPORTED";
        case CLA_ERR_CUDA: return "CLA_ERR_CUDA";
        case CLA_ERR_TIMEOUT: return "CLA_ERR_TIMEOUT";
        case CLA_ERR_WORKSPACE: return "CLA_ERR_WORKSPACE";
        default: return "CLA_ERR_UNKNOWN";
    }
}

extern "C" const char *cla_last_error_message(void) { return cla::g_msg; }

namespace cla {
namespace {
// Waits on a header word that nothing sets: exercises the bounded wait.
__global__ void selftest_wait_kernel(WsHeader *hdr) {
    if (threadIdx.x == 0) (void)wait_flag(&hdr->pad[0], hdr, 99u);
}
}  // namespace
}  // namespace cla

extern "C" int cla_selftest_wait_timeout(void *ws, size_t ws_bytes, void *stream) {
    cla::clear_error();
    if (ws == nullptr || ws_bytes < sizeof(cla::WsHeader) || !cla::aligned16(ws))
        return cla::fail(CLA_ERR_WORKSPACE, "cla_selftest_wait_timeout: need a 16-byte aligned workspace of at least %zu bytes", sizeof(cla::WsHeader));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(cla::WsHeader), s), "cla_selftest_wait_timeout");
    cla::selftest_wait_kernel<<<1, 32, 0, s>>>(static_cast<cla::WsHeader *>(ws));
    return cla::check_launch("cla_selftest_wait_timeout");
}

extern "C" int cla_check_status(const void *ws, void *stream) {
    if (ws == nullptr) return cla::fail(CLA_ERR_INVALID_ARG, "cla_check_status: ws is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cla::WsHeader hdr;
    CLA_CUDA_TRY(cudaMemcpyAsync(&hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost, s), "cla_check_status: copy");
    CLA_CUDA_TRY(cudaStreamSynchronize(s), "cla_check_status: synchronize");
    if (hdr.error & cla::kErrTimeout)
        return cla::fail(CLA_ERR_TIMEOUT, "a cross-block wait gave up (site %u)", hdr.where);
    if (hdr.error & cla::kErrRange)
        return cla::fail(CLA_ERR_UNSUPPORTED,
                         "an input was outside the kernel's range (gated linear attention: a key dimension whose "
                         "decay over 32 tokens of a chunk is below 2^-120, or a zero or non-finite gate; delta "
                         "rule: a non-finite log decay or beta); the results of that call are not valid");
    return CLA_OK;
}

extern "C" int cla_check_device_status(const void *ws, void *stream) { return cla_check_status(ws, stream); }
