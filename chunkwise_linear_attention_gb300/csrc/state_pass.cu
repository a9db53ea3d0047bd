// state_pass.cu -- the two small steps of splitting one sequence across
// devices by state passing ("Parallel Scan", "Splitting one sequence across
// devices"): every device runs its contiguous slice from a zero state, which
// gives the slice's affine pair (alpha_p, dS_p) -- its total decay and its
// own contribution to the state at its end -- and the state entering a slice
// is the composition of the pairs before it under
//     (a1, b1) . (a2, b2) = (a1 a2, a2 b1 + b2),
// applied to the initial state.  The backward runs the same composition from
// the right on the adjoint state.
//   cla_decay_total   alpha = exp(sum over the slice of log a), per head (scalar
//                     decays) or per head and key dimension (gated decays);
//   cla_state_compose folds a list of pairs onto an edge state.
// Both are memory-bound reductions over small arrays; one thread per output
// element, the fold in the list's order (deterministic).
#include "cla_internal.cuh"

namespace cla {
namespace {

constexpr int kPassThreads = 256;

// One block per (head, decay column): the sum of T log decays with stride A.
__global__ void __launch_bounds__(kPassThreads) decay_total_kernel(const float *__restrict__ log_decay,
                                                                   float *__restrict__ alpha, long long T, int A) {
    __shared__ float s_w[kPassThreads / 32];
    const size_t bh = blockIdx.x / (unsigned)A;
    const int a = (int)(blockIdx.x % (unsigned)A);
    const float *src = log_decay + bh * (size_t)T * A + a;
    float acc = 0.f;
    for (long long t = threadIdx.x; t < T; t += kPassThreads) acc += src[(size_t)t * A];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int w = 0; w < kPassThreads / 32; ++w) tot += s_w[w];
        alpha[bh * A + a] = __expf(tot);  // a reset (log a = -inf) anywhere gives 0
    }
}

// out[bh][e] = fold over pairs c = 0..count-1 (pair index j = first + c * step) of
// acc <- alpha[j][bh][e / (n / A)] * acc + dS[j][bh][e], from acc = edge[bh][e] (0 without edge).
__global__ void __launch_bounds__(kPassThreads) state_compose_kernel(const float *__restrict__ alpha,
                                                                     const float *__restrict__ dS,
                                                                     const float *__restrict__ edge,
                                                                     float *__restrict__ out, long long BH, long long n,
                                                                     int A, long long first, long long count,
                                                                     long long step) {
    const long long per = n / A;
    for (long long x = (long long)blockIdx.x * kPassThreads + threadIdx.x; x < BH * n;
         x += (long long)gridDim.x * kPassThreads) {
        const long long bh = x / n, e = x % n;
        float acc = edge ? edge[x] : 0.f;
        for (long long c = 0; c < count; ++c) {
            const long long j = first + c * step;
            acc = fmaf(alpha[(j * BH + bh) * A + e / per], acc, dS[j * BH * n + x]);
        }
        out[x] = acc;
    }
}

}  // namespace
}  // namespace cla

using namespace cla;

extern "C" int cla_decay_total(const float *log_decay, float *alpha, int64_t BH, int64_t T, int64_t A,
                               void *stream) {
    clear_error();
    const char *fn = "cla_decay_total";
    if (BH < 0 || T < 0 || A < 1) return fail(CLA_ERR_INVALID_ARG, "%s: bad sizes", fn);
    if (!product_below({BH, A}, 2147483648.0) || !product_below({BH, T, A}, 9.0e18))
        return fail(CLA_ERR_UNSUPPORTED, "%s: size out of range for one launch", fn);
    if (BH == 0) return CLA_OK;
    if (!alpha || (T > 0 && !log_decay)) return fail(CLA_ERR_INVALID_ARG, "%s: log_decay and alpha required", fn);
    if (!aligned_or_null({log_decay, alpha}, 4)) return fail(CLA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    decay_total_kernel<<<(unsigned int)(BH * A), kPassThreads, 0, s>>>(log_decay, alpha, T, (int)A);
    return check_launch(fn);
}

extern "C" int cla_state_compose(const float *alpha, const float *dS, const float *edge, float *out, int64_t P,
                                 int64_t BH, int64_t n, int64_t A, int64_t first, int64_t count, int64_t step,
                                 void *stream) {
    clear_error();
    const char *fn = "cla_state_compose";
    if (P < 0 || BH < 0 || n < 0 || A < 1 || count < 0 || (n > 0 && n % A != 0))
        return fail(CLA_ERR_INVALID_ARG, "%s: bad sizes (n must be a multiple of A)", fn);
    if (count > 0 && (first < 0 || first >= P || first + (count - 1) * step < 0 || first + (count - 1) * step >= P))
        return fail(CLA_ERR_INVALID_ARG, "%s: pair indices out of range", fn);
    if (!product_below({P, BH, n}, 9.0e18)) return fail(CLA_ERR_UNSUPPORTED, "%s: size out of range", fn);
    if (BH == 0 || n == 0) return CLA_OK;
    if (!out || (count > 0 && (!alpha || !dS))) return fail(CLA_ERR_INVALID_ARG, "%s: alpha, dS, out required", fn);
    if (!aligned_or_null({alpha, dS, edge, out}, 4)) return fail(CLA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long total = BH * n;
    const unsigned int grid = (unsigned int)((total + kPassThreads - 1) / kPassThreads < 152 * 16
                                                 ? (total + kPassThreads - 1) / kPassThreads
                                                 : 152 * 16);
    state_compose_kernel<<<grid, kPassThreads, 0, s>>>(alpha, dS, edge, out, BH, n, (int)A, first, count, step);
    return check_launch(fn);
}
