// delta.cu -- the delta rule with a decay per head (Gated DeltaNet), forward,
// chunkwise, for GB300 (sm_103a).
//
// "Parallel Scan" (zerotofrontier.app), "What one combine costs": the
// transition is the identity minus a rank-one matrix, and a product of such
// matrices is kept as two thin factors (the WY representation); "At real
// scale": the Gated DeltaNet layer, a scalar decay per head besides.  In the
// pages' row convention (S [dk][dv], o_t = q_t S_t):
//     S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t.
//
// Inside a chunk with cumulative decays gamma_r = prod_{u<=r} a_u (from in-
// chunk sums of log a) and the strictly lower triangular
//     A_rs = beta_r (gamma_r / gamma_s) k_r . k_s      (s < r),
// the chunk's writes and corrections fold into
//     X    = diag(beta) (V - diag(gamma) K S)          (S: the incoming state)
//     Veff = (I + A)^-1 X
//     O    = diag(gamma) Q S + ((Q K^T) . D) Veff,  D_rs = gamma_r / gamma_s (s <= r)
//     S'   = gamma_L S + K^T diag(gamma_L / gamma) Veff
// -- decayed linear attention with the values Veff, which depend on the
// incoming state.  (I + A)^-1 is unit lower triangular; it is formed in fp32
// by forward substitution, one column per thread, and kept as two bf16
// parts for its product with X.
//
// This first kernel runs the chunks of a head in order (one block per head
// and 64 value columns, two blocks per SM): the chunk map S -> S' is a dk x dk matrix here, not
// a scalar, so the segment look-back of the other kernels would compose
// matrices; it is not built.  Products on mma.sync m16n8k16 with the operands
// that are not exact bf16 inputs split into two bf16 parts (K S, T X, P Veff,
// the state update), as in the other kernels.
//
// Range: finite log decays (no exact-zero gates).  A chunk with a non-finite
// log decay or gate strength sets an error flag that cla_check_status reports.
#include <algorithm>
#include <type_traits>

#include "cla_internal.cuh"
#include "mma_sync.cuh"

namespace cla {
namespace {

typedef __nv_bfloat16 bf16;

constexpr float kDlLog2e = 1.4426950408889634f;
constexpr int kDlTc = 64;        // tokens per chunk
constexpr int kDlThreads = 128;  // warp w: rows 16w..16w+15 of a chunk
constexpr int kDlBwdThreads = 256;  // backward: warp w rows 16(w & 3).., column half w >> 2
constexpr int kAS = kDlTc + 4;    // row stride (floats) of the fp32 [64][64] triangle: 16-byte aligned rows

// sum_{s < r} row[s] x[s] for the forward substitution of a unit lower triangular 16-row block:
// 16-byte loads of the row (broadcast: the threads of a block read the same row) and four partial
// sums, so the dependent chain per row is a quarter as long.  r is a compile-time constant after
// unrolling; x stays in registers.
__device__ __forceinline__ float tri_row_dot16(const float *row, const float (&x)[16], int r) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int s4 = 0; s4 + 4 <= r; s4 += 4) {
        const float4 e = *reinterpret_cast<const float4 *>(row + s4);
        a0 = fmaf(e.x, x[s4], a0);
        a1 = fmaf(e.y, x[s4 + 1], a1);
        a2 = fmaf(e.z, x[s4 + 2], a2);
        a3 = fmaf(e.w, x[s4 + 3], a3);
    }
#pragma unroll
    for (int s = r & ~3; s < r; ++s) a0 = fmaf(row[s], x[s], a0);
    return (a0 + a1) + (a2 + a3);
}

// Pulls one 128-byte line of global memory into L2 (no register result, no wait).
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// T = (I + A)^-1 in place, A strictly lower triangular, fp32 [64][kAS] in shared memory (zeros on
// and above the diagonal); on return the array holds T (unit diagonal, zeros above).  Blocked by
// 16 rows: the four diagonal blocks T_bb = (I + A_bb)^-1 by forward substitution (threads 0..63,
// one column of one block each), then block rows i = 1, 2, 3 from
//     S_ij = sum_{k=j}^{i-1} A_ik T_kj,   T_ij = -T_ii S_ij      (j < i),
// S in the scratch Sx ([16][48] fp32) and T_ij over A_ij, every thread of the first 128 taking two
// columns of one row.  A dependent chain of 16 rows and three block rows instead of 64 rows.
// Called by the whole block (NT >= 128 threads); ends with a barrier.
__device__ __forceinline__ void tri_inverse_blocked(float *Am, float *Sx, int tid) {
    {  // diagonal blocks
        const int b = (tid >> 4) & 3, c = tid & 15;
        float x[16];
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float acc = tri_row_dot16(Am + (16 * b + r) * kAS + 16 * b, x, r);
                x[r] = (r < c) ? 0.f : (r == c ? 1.f : -acc);
            }
        }
        __syncthreads();  // every diagonal block read
        if (tid < 64) {
#pragma unroll
            for (int r = 0; r < 16; ++r) Am[(16 * b + r) * kAS + 16 * b + c] = x[r];
        }
        __syncthreads();
    }
    constexpr int SXS = 48;                             // row stride of Sx (floats)
    const int r = (tid >> 3) & 15, cp = 2 * (tid & 7);  // this thread's row and column pair in a block
    const bool act = tid < 128;
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        if (act) {
            const float *arow = Am + (16 * i + r) * kAS;
#pragma unroll
            for (int j = 0; j < i; ++j) {
                float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);  // two chains
#pragma unroll
                for (int s4 = 16 * j; s4 < 16 * i; s4 += 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(arow + s4);
                    const float2 t0 = *reinterpret_cast<const float2 *>(Am + (s4 + 0) * kAS + 16 * j + cp);
                    const float2 t1 = *reinterpret_cast<const float2 *>(Am + (s4 + 1) * kAS + 16 * j + cp);
                    const float2 t2 = *reinterpret_cast<const float2 *>(Am + (s4 + 2) * kAS + 16 * j + cp);
                    const float2 t3 = *reinterpret_cast<const float2 *>(Am + (s4 + 3) * kAS + 16 * j + cp);
                    a0 = __ffma2_rn(make_float2(av.x, av.x), t0, a0);
                    a1 = __ffma2_rn(make_float2(av.y, av.y), t1, a1);
                    a0 = __ffma2_rn(make_float2(av.z, av.z), t2, a0);
                    a1 = __ffma2_rn(make_float2(av.w, av.w), t3, a1);
                }
                *reinterpret_cast<float2 *>(Sx + r * SXS + 16 * j + cp) = __fadd2_rn(a0, a1);
            }
        }
        __syncthreads();  // S_i* in the scratch; block row i of A read
        if (act) {
            const float *trow = Am + (16 * i + r) * kAS + 16 * i;  // T_ii, zeros above its diagonal
            float tr[16];
#pragma unroll
            for (int s4 = 0; s4 < 16; s4 += 4) {
                const float4 tv4 = *reinterpret_cast<const float4 *>(trow + s4);
                tr[s4] = tv4.x;
                tr[s4 + 1] = tv4.y;
                tr[s4 + 2] = tv4.z;
                tr[s4 + 3] = tv4.w;
            }
#pragma unroll
            for (int j = 0; j < i; ++j) {
                float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int s = 0; s < 16; s += 2) {
                    a0 = __ffma2_rn(make_float2(tr[s], tr[s]), *reinterpret_cast<const float2 *>(Sx + s * SXS + 16 * j + cp), a0);
                    a1 = __ffma2_rn(make_float2(tr[s + 1], tr[s + 1]),
                                    *reinterpret_cast<const float2 *>(Sx + (s + 1) * SXS + 16 * j + cp), a1);
                }
                const float2 t = __fadd2_rn(a0, a1);
                *reinterpret_cast<float2 *>(Am + (16 * i + r) * kAS + 16 * j + cp) = make_float2(-t.x, -t.y);
            }
        }
        __syncthreads();  // block row i of T in place
    }
}

template <int DK>
struct DeltaCfg {
    static constexpr int QRB = DK * 2;   // bytes per Q / K row (bf16)
    static constexpr int VRB = 128;      // bytes per row of a 64-column slab (bf16)
    static constexpr int Q_BYTES = kDlTc * QRB;
    static constexpr int V_BYTES = kDlTc * VRB;
    // one stage: Q, K, V, log decays, gate strengths
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = 2 * Q_BYTES;
    static constexpr int OFF_L = 2 * Q_BYTES + V_BYTES;
    static constexpr int OFF_B = OFF_L + kDlTc * 4;
    static constexpr int STAGE = OFF_B + kDlTc * 4;
    // Buffers whose lives do not overlap share memory (two blocks then fit an SM):
    // A (fp32) until (I + A)^-1 is built, then X and Veff in the same bytes;
    // (I + A)^-1 until Veff is formed, then diag(gamma_L / gamma) Veff.
    static constexpr int OFF_A = STAGE;                     // A, fp32 [64][64] (row stride 65)
    static constexpr int A_FLOATS = kDlTc * kAS;
    static constexpr int OFF_XH = OFF_A;                    // X, then Veff, two bf16 parts [64][64]
    static constexpr int OFF_XL = OFF_XH + kDlTc * VRB;
    static constexpr int OFF_TH = OFF_A + A_FLOATS * 4;     // (I + A)^-1 as two bf16 parts [64][64]
    static constexpr int OFF_TL = OFF_TH + kDlTc * VRB;
    static constexpr int OFF_WH = OFF_TH;                   // diag(gamma_L / gamma) Veff, two parts
    static constexpr int OFF_WL = OFF_TL;
    static constexpr int OFF_SH = OFF_TL + kDlTc * VRB;     // the state, two bf16 parts [DK][64]
    static constexpr int OFF_SL = OFF_SH + DK * VRB;
    static constexpr int OFF_C = OFF_SL + DK * VRB;         // in-chunk log2 decays c_r [64]
    static constexpr int SMEM = OFF_C + kDlTc * 4;
    static constexpr int S_MT = DK / 64;  // 16-row state tiles per warp
    static_assert(2 * kDlTc * VRB <= A_FLOATS * 4, "X fits where A was");
    static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two blocks per SM");
};

struct DeltaArgs {
    const bf16 *q, *k, *v;
    const float *g, *beta;  // [BH][T]
    const float *S0;        // [BH][DK][DV] or NULL
    float *o, *ST;          // o NULL: the output is not formed (the backward's states pass)
    float *states;          // [BH][n_chunks][DK][DV], the state entering every chunk, or NULL
    // [BH][n_chunks] images of (I + A)^-1 as its two bf16 parts in the swizzled [64][64] tile
    // layout (16 KB per chunk), formed beforehand by delta_wy_kernel; NULL: formed in the chunk loop
    uint8_t *wy;
    // [BH][n_chunks][64][64] fp32 or NULL: E = strictly lower (2^(c_r - c_s) k_r . k_s) of every
    // chunk (A without the gate strengths), written by delta_wy_kernel for the backward
    float *E;
    int BH, DV, nzb, n_chunks;
    long long T;
    WsHeader *hdr;
};

// In-chunk log2 decays c_r (cumulative from the chunk start, one warp) with the range check of
// the chunk's log decays and gate strengths.
__device__ __forceinline__ void delta_chunk_decays(const float *ls, const float *bs, float *cs, int lane,
                                                   WsHeader *hdr) {
    float v0 = ls[2 * lane], v1 = ls[2 * lane + 1];
    const float b0 = bs[2 * lane], b1 = bs[2 * lane + 1];
    if (!isfinite(v0) || !isfinite(v1) || !isfinite(b0) || !isfinite(b1)) atomicOr(&hdr->error, kErrRange);
    v0 *= kDlLog2e;
    v1 = v0 + v1 * kDlLog2e;
    float tot = v1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, tot, off);
        if (lane >= off) tot += o;
    }
    const float ex = tot - v1;  // sum over the earlier lanes' pairs
    cs[2 * lane] = ex + v0;
    cs[2 * lane + 1] = ex + v1;
}

// A = strictly lower (beta_r 2^(c_r - c_s) k_r . k_s) into Am (fp32, row stride kAS): rows
// 16 warp.. of it, K Kt on mma.sync from the swizzled K tile (QRB bytes per row).
template <int DK, int QRB>
__device__ __forceinline__ void delta_build_A(const uint8_t *Kt, const float *bs, const float *cs, float *Am,
                                              int warp, int lane, float *Eg = nullptr) {
    const int g = lane >> 2, tq = lane & 3;
    const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    float F[8][4];
#pragma unroll
    for (int nj = 0; nj < 8; ++nj)
#pragma unroll
        for (int e = 0; e < 4; ++e) F[nj][e] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < DK / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(smem_u32(Kt + swz<QRB>(arow, 2 * kk + (lane >> 4))), a);
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            uint32_t b[4];
            const int brow = 16 * pp + (lane & 7) + (lane >> 4) * 8;
            ldsm_x4(smem_u32(Kt + swz<QRB>(brow, 2 * kk + ((lane >> 3) & 1))), b);
            mma16816(F[2 * pp], a, b[0], b[1]);
            mma16816(F[2 * pp + 1], a, b[2], b[3]);
        }
    }
#pragma unroll
    for (int nj = 0; nj < 8; ++nj)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = warp * 16 + g + 8 * (e >> 1), s = nj * 8 + 2 * tq + (e & 1);
            Am[r * kAS + s] = (s < r) ? bs[r] * ex2(cs[r] - cs[s]) * F[nj][e] : 0.f;
        }
    if (Eg != nullptr) {  // E = A without the gate strengths: the two columns of a pair in one store
#pragma unroll
        for (int nj = 0; nj < 8; ++nj)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = warp * 16 + g + 8 * h, s = nj * 8 + 2 * tq;
                const float e0 = (s < r) ? ex2(cs[r] - cs[s]) * F[nj][2 * h] : 0.f;
                const float e1 = (s + 1 < r) ? ex2(cs[r] - cs[s + 1]) * F[nj][2 * h + 1] : 0.f;
                __stcg(reinterpret_cast<float2 *>(Eg + r * kDlTc + s), make_float2(e0, e1));
            }
    }
}

// T (fp32 in Am, row stride kAS) as two bf16 parts in [64][64] tiles of 128-byte swizzled rows at
// hi and lo (shared or global memory): 16-byte chunks of 8 columns, four per thread.
__device__ __forceinline__ void delta_T_parts(const float *Am, uint8_t *hi_tile, uint8_t *lo_tile, int tid) {
#pragma unroll
    for (int it = 0; it < kDlTc * 8 / kDlThreads; ++it) {
        const int task = tid + it * kDlThreads, r = task >> 3, c8 = task & 7;
        const float4 v0 = *reinterpret_cast<const float4 *>(Am + r * kAS + 8 * c8);
        const float4 v1 = *reinterpret_cast<const float4 *>(Am + r * kAS + 8 * c8 + 4);
        uint32_t hi[4], lo[4];
        split_bf16x2(make_float2(v0.x, v0.y), hi[0], lo[0]);
        split_bf16x2(make_float2(v0.z, v0.w), hi[1], lo[1]);
        split_bf16x2(make_float2(v1.x, v1.y), hi[2], lo[2]);
        split_bf16x2(make_float2(v1.z, v1.w), hi[3], lo[3]);
        *reinterpret_cast<uint4 *>(hi_tile + swz<128>(r, c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(lo_tile + swz<128>(r, c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// The chunks' (I + A)^-1, which do not depend on the state, all at once before the chunk loop:
// one block per (head, chunk), writing the two bf16 parts of each in the tile layout the loop
// copies straight into shared memory.  This takes the K K^T product and the inverse -- about
// half of a chunk's work -- off the loop's sequential path, and forms them once per chunk
// instead of once per 64-column value block.
template <int DK>
__global__ void __launch_bounds__(kDlThreads) delta_wy_kernel(const DeltaArgs p) {
    constexpr int QRB = DK * 2;
    constexpr int OFF_K = 0, OFF_L = kDlTc * QRB, OFF_B = OFF_L + kDlTc * 4, OFF_C = OFF_B + kDlTc * 4;
    constexpr int OFF_A = OFF_C + kDlTc * 4, OFF_S = OFF_A + kDlTc * kAS * 4;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / p.n_chunks, chunk = blockIdx.x % p.n_chunks;
    const long long t0 = (long long)chunk * kDlTc;
    const bf16 *Kb = p.k + (size_t)bh * p.T * DK;
    constexpr int QC = QRB / 16;
    for (int i = tid; i < kDlTc * QC; i += kDlThreads) {
        const int row = i / QC, c16 = i % QC;
        const long long t = t0 + row;
        const bool ok = t < p.T;
        cp_async16(smem_u32(smem + OFF_K + swz<QRB>(row, c16)), Kb + (size_t)(ok ? t : 0) * DK + c16 * 8,
                   ok ? 16u : 0u);
    }
    for (int i = tid; i < kDlTc; i += kDlThreads) {  // padding tokens: no decay, no write
        const long long t = t0 + i;
        const bool ok = t < p.T;
        cp_async4(smem_u32(smem + OFF_L + i * 4), p.g + (size_t)bh * p.T + (ok ? t : 0), ok ? 4u : 0u);
        cp_async4(smem_u32(smem + OFF_B + i * 4), p.beta + (size_t)bh * p.T + (ok ? t : 0), ok ? 4u : 0u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    const float *bs = reinterpret_cast<const float *>(smem + OFF_B);
    float *cs = reinterpret_cast<float *>(smem + OFF_C);
    float *Am = reinterpret_cast<float *>(smem + OFF_A);
    if (warp == 0) delta_chunk_decays(reinterpret_cast<const float *>(smem + OFF_L), bs, cs, lane, p.hdr);
    __syncthreads();
    delta_build_A<DK, QRB>(smem + OFF_K, bs, cs, Am, warp, lane,
                           p.E != nullptr ? p.E + ((size_t)bh * p.n_chunks + chunk) * (kDlTc * kDlTc) : nullptr);
    __syncthreads();
    tri_inverse_blocked(Am, reinterpret_cast<float *>(smem + OFF_S), tid);
    uint8_t *out = p.wy + ((size_t)bh * p.n_chunks + chunk) * (2 * kDlTc * 128);
    delta_T_parts(Am, out, out + kDlTc * 128, tid);
}
constexpr int delta_wy_smem(int DK) { return kDlTc * DK * 2 + 3 * kDlTc * 4 + kDlTc * kAS * 4 + 16 * 48 * 4; }

template <int DK>
__global__ void __launch_bounds__(kDlThreads, 2) delta_fwd_kernel(const DeltaArgs p) {
    using C = DeltaCfg<DK>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int bh = blockIdx.x / p.nzb, zb = blockIdx.x % p.nzb;
    const bf16 *Qb = p.q + (size_t)bh * p.T * DK;
    const bf16 *Kb = p.k + (size_t)bh * p.T * DK;
    const bf16 *Vb = p.v + (size_t)bh * p.T * p.DV + zb * 64;
    const float *Lb = p.g + (size_t)bh * p.T;
    const float *Bb = p.beta + (size_t)bh * p.T;
    float *Am = reinterpret_cast<float *>(smem + C::OFF_A);
    float *cs = reinterpret_cast<float *>(smem + C::OFF_C);

    auto load_stage = [&](int stage, int chunk) {
        uint8_t *st = smem + stage * C::STAGE;
        const long long t0 = (long long)chunk * kDlTc;
        constexpr int QC = C::QRB / 16;
        for (int i = tid; i < kDlTc * QC; i += kDlThreads) {
            const int row = i / QC, c16 = i % QC;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            const size_t off = (size_t)(ok ? t : 0) * DK + c16 * 8;
            cp_async16(smem_u32(st + C::OFF_Q + swz<C::QRB>(row, c16)), Qb + off, ok ? 16u : 0u);
            cp_async16(smem_u32(st + C::OFF_K + swz<C::QRB>(row, c16)), Kb + off, ok ? 16u : 0u);
        }
        for (int i = tid; i < kDlTc * 8; i += kDlThreads) {
            const int row = i >> 3, c16 = i & 7;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            cp_async16(smem_u32(st + C::OFF_V + swz<C::VRB>(row, c16)), Vb + (size_t)(ok ? t : 0) * p.DV + c16 * 8,
                       ok ? 16u : 0u);
        }
        for (int i = tid; i < kDlTc; i += kDlThreads) {  // padding tokens: no decay, no write
            const long long t = t0 + i;
            const bool ok = t < p.T;
            cp_async4(smem_u32(st + C::OFF_L + i * 4), Lb + (ok ? t : 0), ok ? 4u : 0u);
            cp_async4(smem_u32(st + C::OFF_B + i * 4), Bb + (ok ? t : 0), ok ? 4u : 0u);
        }
        if (p.wy != nullptr) {  // the chunk's (I + A)^-1 parts: 16 KB copied as they lie
            const uint8_t *src = p.wy + ((size_t)bh * p.n_chunks + chunk) * (2 * kDlTc * 128);
            for (int i = tid; i < 2 * kDlTc * 8; i += kDlThreads)
                cp_async16(smem_u32(smem + C::OFF_TH + 16 * i), src + 16 * i, 16u);
        }
    };
    // state fragments: warp w owns rows 16(w S_MT + mi) + {g, g + 8}
    constexpr int S_MT = C::S_MT;
    float S[S_MT][8][4];
    auto s_row = [&](int mi, int h) { return (warp * S_MT + mi) * 16 + g + 8 * h; };
#pragma unroll
    for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
        for (int nj = 0; nj < 8; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                S[mi][nj][e] = p.S0 ? __ldg(p.S0 + ((size_t)bh * DK + s_row(mi, e >> 1)) * p.DV + zb * 64 + nj * 8 +
                                            2 * tq + (e & 1))
                                    : 0.f;
    // a [64][64] tile of fp32 fragments (this warp's 16 rows) into two bf16 tiles, [row][col]
    auto store_parts = [&](const float (&F)[8][4], int off_hi, int off_lo, int row0) {
#pragma unroll
        for (int nj = 0; nj < 8; ++nj)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = row0 + g + 8 * h, col = nj * 8 + 2 * tq;
                const uint32_t off = swz<C::VRB>(row, col >> 3) + (col & 7) * 2;
                uint32_t hi, lo;
                split_bf16x2(make_float2(F[nj][2 * h], F[nj][2 * h + 1]), hi, lo);
                *reinterpret_cast<uint32_t *>(smem + off_hi + off) = hi;
                *reinterpret_cast<uint32_t *>(smem + off_lo + off) = lo;
            }
    };
    auto write_state_parts = [&]() {
#pragma unroll
        for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = s_row(mi, h), col = nj * 8 + 2 * tq;
                    const uint32_t off = swz<C::VRB>(row, col >> 3) + (col & 7) * 2;
                    uint32_t hi, lo;
                    split_bf16x2(make_float2(S[mi][nj][2 * h], S[mi][nj][2 * h + 1]), hi, lo);
                    *reinterpret_cast<uint32_t *>(smem + C::OFF_SH + off) = hi;
                    *reinterpret_cast<uint32_t *>(smem + C::OFF_SL + off) = lo;
                }
    };
    // F += (rows 16w.. of an A operand tile [64][K] at a_off, K = 16 kk) x (B [K][64] via trans)
    auto zero8 = [&](float (&F)[8][4]) {
#pragma unroll
        for (int nj = 0; nj < 8; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e) F[nj][e] = 0.f;
    };
    const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;

    // one stage of loads: the next chunk's is issued once this chunk's inputs are consumed (a
    // second block on the SM runs meanwhile)
    load_stage(0, 0);
    cp_async_commit();
    for (int i = 0; i < p.n_chunks; ++i) {
        const int stage = 0;
        uint8_t *st = smem;
        const float *ls = reinterpret_cast<const float *>(st + C::OFF_L);
        const float *bs = reinterpret_cast<const float *>(st + C::OFF_B);
        const long long t0 = (long long)i * kDlTc;
        if (p.states != nullptr) {  // the state entering chunk i, for the backward
            float *sg = p.states + ((size_t)bh * p.n_chunks + i) * DK * p.DV + zb * 64;
#pragma unroll
            for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
                for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        __stcg(reinterpret_cast<float2 *>(sg + (size_t)s_row(mi, h) * p.DV + nj * 8 + 2 * tq),
                               make_float2(S[mi][nj][2 * h], S[mi][nj][2 * h + 1]));
        }
        cp_async_wait<0>();
        __syncthreads();
        // ---- in-chunk log2 decays (warp 0) and the state's bf16 parts (everyone)
        if (warp == 0) delta_chunk_decays(ls, bs, cs, lane, p.hdr);
        write_state_parts();
        __syncthreads();
        const float cL = cs[kDlTc - 1];

        if (p.wy == nullptr) {
            // ---- A = strictly lower (beta_r 2^(c_r - c_s) k_r . k_s), this warp's 16 rows
            delta_build_A<DK, C::QRB>(st + C::OFF_K, bs, cs, Am, warp, lane);
            __syncthreads();
            // ---- T = (I + A)^-1 (unit lower triangular) in place (scratch: T's tiles, free until
            // below), then as two bf16 parts in the [64][64] tiles
            tri_inverse_blocked(Am, reinterpret_cast<float *>(smem + C::OFF_TH), tid);
            delta_T_parts(Am, smem + C::OFF_TH, smem + C::OFF_TL, tid);
            __syncthreads();
        }

        // ---- X = diag(beta) (V - diag(gamma) K S) for this warp's rows (K S: two products)
        {
            float F[8][4];
            zero8(F);
#pragma unroll 2
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t a[4];
                ldsm_x4(smem_u32(st + C::OFF_K + swz<C::QRB>(arow, 2 * kk + (lane >> 4))), a);
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const int brow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t boff = swz<C::VRB>(brow, 2 * pp + (lane >> 4));
                    uint32_t sh[4], sl[4];
                    ldsm_x4_t(smem_u32(smem + C::OFF_SH + boff), sh);
                    ldsm_x4_t(smem_u32(smem + C::OFF_SL + boff), sl);
                    mma16816(F[2 * pp], a, sh[0], sh[1]);
                    mma16816(F[2 * pp + 1], a, sh[2], sh[3]);
                    mma16816(F[2 * pp], a, sl[0], sl[1]);
                    mma16816(F[2 * pp + 1], a, sl[2], sl[3]);
                }
            }
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = warp * 16 + g + 8 * h, col = nj * 8 + 2 * tq;
                    const float2 vv = unpack_bf16(
                        *reinterpret_cast<const uint32_t *>(st + C::OFF_V + swz<C::VRB>(r, col >> 3) + (col & 7) * 2));
                    const float gm = ex2(cs[r]), bt = bs[r];
                    F[nj][2 * h] = bt * (vv.x - gm * F[nj][2 * h]);
                    F[nj][2 * h + 1] = bt * (vv.y - gm * F[nj][2 * h + 1]);
                }
            store_parts(F, C::OFF_XH, C::OFF_XL, warp * 16);
        }
        __syncthreads();

        // ---- Veff = T X (three products), then Veff and diag(gamma_L / gamma) Veff as bf16 parts
        {
            float F[8][4];
            zero8(F);
#pragma unroll
            for (int kt = 0; kt < kDlTc / 16; ++kt) {
                uint32_t th[4], tl[4];
                const uint32_t aoff = swz<C::VRB>(arow, 2 * kt + (lane >> 4));
                ldsm_x4(smem_u32(smem + C::OFF_TH + aoff), th);
                ldsm_x4(smem_u32(smem + C::OFF_TL + aoff), tl);
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const int brow = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t boff = swz<C::VRB>(brow, 2 * pp + (lane >> 4));
                    uint32_t xh[4], xl[4];
                    ldsm_x4_t(smem_u32(smem + C::OFF_XH + boff), xh);
                    ldsm_x4_t(smem_u32(smem + C::OFF_XL + boff), xl);
                    mma16816(F[2 * pp], th, xh[0], xh[1]);
                    mma16816(F[2 * pp + 1], th, xh[2], xh[3]);
                    mma16816(F[2 * pp], th, xl[0], xl[1]);
                    mma16816(F[2 * pp + 1], th, xl[2], xl[3]);
                    mma16816(F[2 * pp], tl, xh[0], xh[1]);
                    mma16816(F[2 * pp + 1], tl, xh[2], xh[3]);
                }
            }
            __syncthreads();  // every warp has read X
            store_parts(F, C::OFF_XH, C::OFF_XL, warp * 16);
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float w = ex2(cL - cs[warp * 16 + g + 8 * h]);
                    F[nj][2 * h] *= w;
                    F[nj][2 * h + 1] *= w;
                }
            store_parts(F, C::OFF_WH, C::OFF_WL, warp * 16);
        }
        __syncthreads();

        // ---- O = diag(gamma) Q S + ((Q K^T) . D) Veff
        if (p.o != nullptr) {
            float O[8][4], P[8][4];
            zero8(O);
            zero8(P);
#pragma unroll 2
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t a[4];
                ldsm_x4(smem_u32(st + C::OFF_Q + swz<C::QRB>(arow, 2 * kk + (lane >> 4))), a);
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const int brow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t boff = swz<C::VRB>(brow, 2 * pp + (lane >> 4));
                    uint32_t sh[4], sl[4];
                    ldsm_x4_t(smem_u32(smem + C::OFF_SH + boff), sh);
                    ldsm_x4_t(smem_u32(smem + C::OFF_SL + boff), sl);
                    mma16816(O[2 * pp], a, sh[0], sh[1]);
                    mma16816(O[2 * pp + 1], a, sh[2], sh[3]);
                    mma16816(O[2 * pp], a, sl[0], sl[1]);
                    mma16816(O[2 * pp + 1], a, sl[2], sl[3]);
                    uint32_t kb[4];
                    const int krow = 16 * pp + (lane & 7) + (lane >> 4) * 8;
                    ldsm_x4(smem_u32(st + C::OFF_K + swz<C::QRB>(krow, 2 * kk + ((lane >> 3) & 1))), kb);
                    mma16816(P[2 * pp], a, kb[0], kb[1]);
                    mma16816(P[2 * pp + 1], a, kb[2], kb[3]);
                }
            }
            uint32_t ph[4][4], pl[4][4];
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = warp * 16 + g + 8 * h, s0 = nj * 8 + 2 * tq;
                    const float gm = ex2(cs[r]);
                    O[nj][2 * h] *= gm;
                    O[nj][2 * h + 1] *= gm;
                    const float x0 = (s0 <= r) ? P[nj][2 * h] * ex2(cs[r] - cs[s0]) : 0.f;
                    const float x1 = (s0 + 1 <= r) ? P[nj][2 * h + 1] * ex2(cs[r] - cs[s0 + 1]) : 0.f;
                    split_bf16x2(make_float2(x0, x1), ph[nj >> 1][(nj & 1) * 2 + h], pl[nj >> 1][(nj & 1) * 2 + h]);
                }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const int brow = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t boff = swz<C::VRB>(brow, 2 * pp + (lane >> 4));
                    uint32_t vh[4], vl[4];
                    ldsm_x4_t(smem_u32(smem + C::OFF_XH + boff), vh);
                    ldsm_x4_t(smem_u32(smem + C::OFF_XL + boff), vl);
                    mma16816(O[2 * pp], ph[kt], vh[0], vh[1]);
                    mma16816(O[2 * pp + 1], ph[kt], vh[2], vh[3]);
                    mma16816(O[2 * pp], ph[kt], vl[0], vl[1]);
                    mma16816(O[2 * pp + 1], ph[kt], vl[2], vl[3]);
                    mma16816(O[2 * pp], pl[kt], vh[0], vh[1]);
                    mma16816(O[2 * pp + 1], pl[kt], vh[2], vh[3]);
                }
            }
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long t = t0 + warp * 16 + g + 8 * h;
                    if (t < p.T)
                        *reinterpret_cast<float2 *>(p.o + ((size_t)bh * p.T + t) * p.DV + zb * 64 + nj * 8 + 2 * tq) =
                            make_float2(O[nj][2 * h], O[nj][2 * h + 1]);
                }
        }

        // ---- S = gamma_L S + K^T (diag(gamma_L / gamma) Veff)   (two products)
        {
            const float gL = ex2(cL);
#pragma unroll
            for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
                for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                    for (int e = 0; e < 4; ++e) S[mi][nj][e] *= gL;
#pragma unroll
            for (int kt = 0; kt < kDlTc / 16; ++kt) {
                uint32_t b[4][4], bl[4][4];
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const int brow = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t boff = swz<C::VRB>(brow, 2 * pp + (lane >> 4));
                    ldsm_x4_t(smem_u32(smem + C::OFF_WH + boff), b[pp]);
                    ldsm_x4_t(smem_u32(smem + C::OFF_WL + boff), bl[pp]);
                }
#pragma unroll
                for (int mi = 0; mi < S_MT; ++mi) {
                    const int kr = kt * 16 + (lane & 7) + (lane >> 4) * 8;
                    const int kc16 = 2 * (warp * S_MT + mi) + ((lane >> 3) & 1);
                    uint32_t a[4];
                    ldsm_x4_t(smem_u32(st + C::OFF_K + swz<C::QRB>(kr, kc16)), a);
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        mma16816(S[mi][2 * pp], a, b[pp][0], b[pp][1]);
                        mma16816(S[mi][2 * pp + 1], a, b[pp][2], b[pp][3]);
                        mma16816(S[mi][2 * pp], a, bl[pp][0], bl[pp][1]);
                        mma16816(S[mi][2 * pp + 1], a, bl[pp][2], bl[pp][3]);
                    }
                }
            }
        }
        __syncthreads();
        if (i + 1 < p.n_chunks) load_stage(stage, i + 1);
        cp_async_commit();
    }
    cp_async_wait<0>();
    if (p.ST != nullptr) {
#pragma unroll
        for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    p.ST[((size_t)bh * DK + s_row(mi, e >> 1)) * p.DV + zb * 64 + nj * 8 + 2 * tq + (e & 1)] =
                        S[mi][nj][e];
    }
}

template <int DK>
int launch_delta_wy(const DeltaArgs &a, cudaStream_t s) {
    const size_t blocks = (size_t)a.BH * a.n_chunks;
    if (blocks >= 2147483648ull) return fail(CLA_ERR_UNSUPPORTED, "delta_wy_kernel: too many chunks for one launch");
    static std::atomic<unsigned long long> smem_set{0};
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(delta_wy_kernel<DK>), delta_wy_smem(DK));
    if (st) return st;
    delta_wy_kernel<DK><<<(unsigned int)blocks, kDlThreads, delta_wy_smem(DK), s>>>(a);
    return check_launch("delta_wy_kernel");
}

template <int DK>
int launch_delta_fwd(const DeltaArgs &a, cudaStream_t s, unsigned int grid) {
    using C = DeltaCfg<DK>;
    static std::atomic<unsigned long long> smem_set{0};
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(delta_fwd_kernel<DK>), C::SMEM);
    if (st) return st;
    delta_fwd_kernel<DK><<<grid, kDlThreads, C::SMEM, s>>>(a);
    return check_launch("delta_fwd_kernel");
}

// Operand loaders of m16n8k16 from XOR-swizzled row-major tiles (RB bytes per row).
// A operand: 16 rows from row0, k-step kk, of the tile itself.
template <int RB>
__device__ __forceinline__ void lda_rows(uint32_t (&a)[4], const uint8_t *t, int row0, int kk, int lane) {
    ldsm_x4(smem_u32(t + swz<RB>(row0 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * kk + (lane >> 4))), a);
}
// A operand: rows 16 mt.. of the transpose of a tile stored [k][m], k-step kk.
template <int RB>
__device__ __forceinline__ void lda_trans(uint32_t (&a)[4], const uint8_t *t, int mt, int kk, int lane) {
    ldsm_x4_t(smem_u32(t + swz<RB>(kk * 16 + (lane & 7) + (lane >> 4) * 8, 2 * mt + ((lane >> 3) & 1))), a);
}
// B operands of the n-tiles 2pp and 2pp + 1 at k-step kk, B[k][n] = tile[n][k].
template <int RB>
__device__ __forceinline__ void ldb_nk(uint32_t (&b)[4], const uint8_t *t, int pp, int kk, int lane) {
    ldsm_x4(smem_u32(t + swz<RB>(16 * pp + (lane & 7) + (lane >> 4) * 8, 2 * kk + ((lane >> 3) & 1))), b);
}
// The same with B[k][n] = tile[k][n].
template <int RB>
__device__ __forceinline__ void ldb_kn(uint32_t (&b)[4], const uint8_t *t, int pp, int kk, int lane) {
    ldsm_x4_t(smem_u32(t + swz<RB>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * pp + (lane >> 4))), b);
}
template <int N>
__device__ __forceinline__ void mma_pair(float (&F)[N][4], int pp, const uint32_t (&a)[4], const uint32_t (&b)[4]) {
    mma16816(F[2 * pp], a, b[0], b[1]);
    mma16816(F[2 * pp + 1], a, b[2], b[3]);
}
// Sum over the four lanes of a quad (the lanes holding one accumulator row).
__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// ------------------------------------------------------------------ backward
// The adjoint of the chunk form, chunks of a head in reverse, from the state
// entering every chunk (written by the forward kernel's states pass).  Per
// chunk, with P = (Q K^T) . D, E_rs = D_rs k_r . k_s (s < r), A = diag(beta) E,
// U = (I + A)^-1 X, w_r = gamma_L / gamma_r and dS' the adjoint of the state
// leaving the chunk:
//     dU = P^T dO + diag(w) K dS'          dX = (I + A)^-T dU     dV = diag(beta) dX
//     dP = dO U^T (s <= r)                 dA = -dX U^T (s < r)   F  = diag(beta) dA . D
//     dQ = (dP . D) K + diag(gamma) dO S^T
//     dK = (dP . D)^T Q + (F + F^T) K + diag(w) U dS'^T - diag(beta gamma) dX S^T
//     dbeta_r = (V - diag(gamma) K S)_r . dX_r + sum_s dA_rs E_rs
//     dS = gamma_L dS' + Q^T diag(gamma) dO - K^T diag(beta gamma) dX
// and the gradient on the in-chunk log-decay sums c: every decay ratio
// exp(c_r - c_s) differentiated in c (row sums minus column sums of
// dP . P and dA . A), gamma_r q_r . (dO S^T)_r, -beta_r gamma_r (K S)_r . dX_r,
// -w_r (K dS')_r . U_r, and at the chunk's last position
// sum_r w_r (K dS')_r . U_r + gamma_L <S, dS'>; its suffix sums inside the
// chunk are the gradient on each token's log decay.
//
// One block per (head, 64 value columns), 8 warps: warp w takes the chunk's rows
// 16(w & 3)..+15 and half (w >> 2) of the output columns of every product (the
// score-shaped products whose result feeds another product's k dimension are
// formed whole by both warps of a row group, or pass through shared memory);
// the adjoint state dS [DK][64] in registers, split the same way.  dQ, dK, dbeta and dlog_a sum over the value-column blocks: the block
// of columns 0..63 writes them to the outputs, the others to workspace
// partials that delta_bwd_reduce_kernel adds.  dV and dS0 belong to one block.
template <int DK>
struct DeltaBwdCfg {
    static constexpr int QRB = DK * 2;  // bytes per Q / K row
    static constexpr int VRB = 128;     // bytes per row of a [..][64] bf16 tile
    static constexpr int Q_BYTES = kDlTc * QRB;
    static constexpr int V_BYTES = kDlTc * VRB;
    static constexpr int S_BYTES = DK * VRB;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + Q_BYTES;
    static constexpr int OFF_DO = OFF_V + V_BYTES;
    static constexpr int OFF_L = OFF_DO + V_BYTES;   // log decays [64]
    static constexpr int OFF_B = OFF_L + 256;        // gate strengths [64]
    static constexpr int OFF_C = OFF_B + 256;        // in-chunk log2 decays c_r [64]
    static constexpr int OFF_SH = OFF_C + 256;       // S entering the chunk, two bf16 parts [DK][64]
    static constexpr int OFF_SL = OFF_SH + S_BYTES;
    static constexpr int OFF_GH = OFF_SL + S_BYTES;  // dS' (adjoint of the state leaving it), two parts
    static constexpr int OFF_GL = OFF_GH + S_BYTES;
    static constexpr int OFF_E = OFF_GL + S_BYTES;   // E fp32 [64][65]; then F as two parts
    static constexpr int E_BYTES = kDlTc * kAS * 4;
    static constexpr int OFF_FH = OFF_E;
    static constexpr int OFF_FL = OFF_E + V_BYTES;
    static constexpr int OFF_TH = OFF_E + E_BYTES;   // (I + A)^-1; then diag(gamma) dO (two parts each)
    static constexpr int OFF_TL = OFF_TH + V_BYTES;
    static constexpr int OFF_XH = OFF_TL + V_BYTES;  // X; then dU; then dP . D
    static constexpr int OFF_XL = OFF_XH + V_BYTES;
    static constexpr int OFF_UH = OFF_XL + V_BYTES;  // U
    static constexpr int OFF_UL = OFF_UH + V_BYTES;
    static constexpr int OFF_WH = OFF_UL + V_BYTES;  // diag(w) U
    static constexpr int OFF_WL = OFF_WH + V_BYTES;
    static constexpr int OFF_ZH = OFF_WL + V_BYTES;  // -diag(beta gamma) dX
    static constexpr int OFF_ZL = OFF_ZH + V_BYTES;
    static constexpr int OFF_ROW = OFF_ZL + V_BYTES;  // row parts of the gradient on c [2][64]
    static constexpr int OFF_COL = OFF_ROW + 512;     // column parts, one row per warp [8][64]
    static constexpr int OFF_DB = OFF_COL + 2048;     // dbeta parts [2][64]
    static constexpr int OFF_RED = OFF_DB + 512;      // the last position's extra term, per warp [8]
    static constexpr int SMEM = OFF_RED + 64;
    static constexpr int S_MT = DK / 64;  // 16-row tiles of the state per row group
    static_assert(2 * V_BYTES <= E_BYTES, "F fits where E was");
    static_assert(E_BYTES + 16 * 48 * 4 <= 4 * V_BYTES, "the fp32 inverse and its scratch fit over U's tiles");
    static_assert(E_BYTES % 128 == 0, "tiles after E stay 128-byte aligned");
    static_assert(SMEM + 1024 <= 227 * 1024, "one block per SM");
};

struct DeltaBwdArgs {
    const bf16 *q, *k, *v, *dO;
    const float *g, *beta;  // [BH][T]
    const float *dST;       // [BH][DK][DV] or NULL
    const float *states;    // [BH][n_chunks][DK][DV]
    const uint8_t *wy;      // [BH][n_chunks] (I + A)^-1 parts, as delta_wy_kernel writes them
    const float *E;         // [BH][n_chunks][64][64]: the chunks' E, as delta_wy_kernel writes it
    float *dq, *dk, *dv, *dlog, *dbeta, *dS0;
    float *part;            // partials of the column blocks 1.. (NULL when DV == 64)
    long long part_stride;  // floats per column block: BH T (2 DK + 2)
    int BH, DV, nzb, n_chunks;
    long long T;
};

template <int DK>
__global__ void __launch_bounds__(kDlBwdThreads, 1) delta_bwd_kernel(const DeltaBwdArgs p) {
    using C = DeltaBwdCfg<DK>;
    constexpr int S_MT = C::S_MT;
    constexpr int NQ2 = DK / 16;  // 8-column tiles of this warp's half of a [..][DK] output
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int wr = warp & 3, hf = warp >> 2;  // row group, column half
    const int bh = blockIdx.x / p.nzb, zb = blockIdx.x % p.nzb;
    const size_t tok0 = (size_t)bh * p.T;
    const bf16 *Qb = p.q + tok0 * DK;
    const bf16 *Kb = p.k + tok0 * DK;
    const bf16 *Vb = p.v + tok0 * p.DV + zb * 64;
    const bf16 *dOb = p.dO + tok0 * p.DV + zb * 64;
    const float *Lb = p.g + tok0;
    const float *Bb = p.beta + tok0;
    float *dq_out, *dk_out, *dl_out, *db_out;
    if (zb == 0) {
        dq_out = p.dq + tok0 * DK;
        dk_out = p.dk + tok0 * DK;
        dl_out = p.dlog + tok0;
        db_out = p.dbeta + tok0;
    } else {
        float *base = p.part + (size_t)(zb - 1) * p.part_stride;
        const size_t ntok = (size_t)p.BH * p.T;
        dq_out = base + tok0 * DK;
        dk_out = base + ntok * DK + tok0 * DK;
        dl_out = base + 2 * ntok * DK + tok0;
        db_out = base + 2 * ntok * DK + ntok + tok0;
    }
    float *Em = reinterpret_cast<float *>(smem + C::OFF_E);
    float *cs = reinterpret_cast<float *>(smem + C::OFF_C);
    const float *ls = reinterpret_cast<const float *>(smem + C::OFF_L);
    const float *bs = reinterpret_cast<const float *>(smem + C::OFF_B);
    float *rowp = reinterpret_cast<float *>(smem + C::OFF_ROW);  // [2][64]: per column half
    float *colp = reinterpret_cast<float *>(smem + C::OFF_COL);  // [8][64]: per warp, its half's columns
    float *dbs = reinterpret_cast<float *>(smem + C::OFF_DB);    // [2][64]
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);   // [8]
    const uint8_t *sQ = smem + C::OFF_Q, *sK = smem + C::OFF_K, *sdO = smem + C::OFF_DO;
    constexpr int QRB = C::QRB, VRB = C::VRB;
    constexpr int KQ = DK / 16;  // k-steps over the key dimension

    auto load_stage = [&](int chunk) {
        const long long t0 = (long long)chunk * kDlTc;
        constexpr int QC = C::QRB / 16;
        for (int i = tid; i < kDlTc * QC; i += kDlBwdThreads) {
            const int row = i / QC, c16 = i % QC;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            const size_t off = (size_t)(ok ? t : 0) * DK + c16 * 8;
            cp_async16(smem_u32(smem + C::OFF_Q + swz<C::QRB>(row, c16)), Qb + off, ok ? 16u : 0u);
            cp_async16(smem_u32(smem + C::OFF_K + swz<C::QRB>(row, c16)), Kb + off, ok ? 16u : 0u);
        }
        for (int i = tid; i < kDlTc * 8; i += kDlBwdThreads) {
            const int row = i >> 3, c16 = i & 7;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            const size_t off = (size_t)(ok ? t : 0) * p.DV + c16 * 8;
            cp_async16(smem_u32(smem + C::OFF_V + swz<C::VRB>(row, c16)), Vb + off, ok ? 16u : 0u);
            cp_async16(smem_u32(smem + C::OFF_DO + swz<C::VRB>(row, c16)), dOb + off, ok ? 16u : 0u);
        }
        for (int i = tid; i < kDlTc; i += kDlBwdThreads) {  // padding tokens: no decay, no write
            const long long t = t0 + i;
            const bool ok = t < p.T;
            cp_async4(smem_u32(smem + C::OFF_L + i * 4), Lb + (ok ? t : 0), ok ? 4u : 0u);
            cp_async4(smem_u32(smem + C::OFF_B + i * 4), Bb + (ok ? t : 0), ok ? 4u : 0u);
        }
        {  // the chunk's (I + A)^-1 parts and E, formed by delta_wy_kernel (E into rows of kAS floats)
            const uint8_t *src = p.wy + ((size_t)bh * p.n_chunks + chunk) * (2 * kDlTc * 128);
            for (int i = tid; i < 2 * kDlTc * 8; i += kDlBwdThreads)
                cp_async16(smem_u32(smem + C::OFF_TH + 16 * i), src + 16 * i, 16u);
            const float *esrc = p.E + ((size_t)bh * p.n_chunks + chunk) * (kDlTc * kDlTc);
            for (int i = tid; i < kDlTc * 16; i += kDlBwdThreads) {
                const int r = i >> 4, c4 = i & 15;
                cp_async16(smem_u32(smem + C::OFF_E + (r * kAS + 4 * c4) * 4), esrc + r * kDlTc + 4 * c4, 16u);
            }
        }
        // the state entering the chunk, fp32 -> two bf16 parts (plain loads, read once; all of a
        // thread's loads issued before the first is used)
        const float *sg = p.states + ((size_t)bh * p.n_chunks + chunk) * DK * p.DV + zb * 64;
        float4 xs[DK * 16 / kDlBwdThreads];
#pragma unroll
        for (int it = 0; it < DK * 16 / kDlBwdThreads; ++it) {
            const int i = tid + it * kDlBwdThreads, row = i >> 4, c4 = i & 15;
            xs[it] = __ldcs(reinterpret_cast<const float4 *>(sg + (size_t)row * p.DV + c4 * 4));
        }
#pragma unroll
        for (int it = 0; it < DK * 16 / kDlBwdThreads; ++it) {
            const int i = tid + it * kDlBwdThreads, row = i >> 4, c4 = i & 15;
            const float4 x = xs[it];
            uint2 hi, lo;
            split_bf16x2(make_float2(x.x, x.y), hi.x, lo.x);
            split_bf16x2(make_float2(x.z, x.w), hi.y, lo.y);
            const uint32_t off = swz<C::VRB>(row, c4 >> 1) + (c4 & 1) * 8;
            *reinterpret_cast<uint2 *>(smem + C::OFF_SH + off) = hi;
            *reinterpret_cast<uint2 *>(smem + C::OFF_SL + off) = lo;
        }
    };
    // the lines load_stage(chunk) reads, pulled into L2 one chunk ahead (three or so a thread)
    auto prefetch_stage = [&](int chunk) {
        const long long t0 = (long long)chunk * kDlTc;
        const int nrow = (int)min((long long)kDlTc, p.T - t0);
        constexpr int QL = C::QRB / 128;  // 128-byte lines of a Q / K row
        for (int i = tid; i < nrow * QL; i += kDlBwdThreads) {
            const size_t off = (size_t)(t0 + i / QL) * DK + (i % QL) * 64;
            prefetch_l2(Qb + off);
            prefetch_l2(Kb + off);
        }
        for (int i = tid; i < nrow; i += kDlBwdThreads) {
            prefetch_l2(Vb + (size_t)(t0 + i) * p.DV);
            prefetch_l2(dOb + (size_t)(t0 + i) * p.DV);
        }
        if (tid < 2 && 32 * tid < nrow) {
            prefetch_l2(Lb + t0 + 32 * tid);
            prefetch_l2(Bb + t0 + 32 * tid);
        }
        const float *sg = p.states + ((size_t)bh * p.n_chunks + chunk) * DK * p.DV + zb * 64;
        for (int i = tid; i < DK * 2; i += kDlBwdThreads) prefetch_l2(sg + (size_t)(i >> 1) * p.DV + (i & 1) * 32);
        const uint8_t *wy = p.wy + ((size_t)bh * p.n_chunks + chunk) * (2 * kDlTc * 128);
        for (int i = tid; i < 2 * kDlTc; i += kDlBwdThreads) prefetch_l2(wy + 128 * i);
        const float *eg = p.E + ((size_t)bh * p.n_chunks + chunk) * (kDlTc * kDlTc);
        for (int i = tid; i < kDlTc * 2; i += kDlBwdThreads) prefetch_l2(eg + 32 * i);
    };

    // adjoint state fragments: rows 16(wr S_MT + mi) + {g, g + 8}, columns 8(4 hf + nj) + 2 tq + {0, 1}
    float dS[S_MT][4][4];
    auto s_row = [&](int mi, int h) { return (wr * S_MT + mi) * 16 + g + 8 * h; };
#pragma unroll
    for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dS[mi][nj][e] = p.dST ? __ldg(p.dST + ((size_t)bh * DK + s_row(mi, e >> 1)) * p.DV + zb * 64 +
                                              (4 * hf + nj) * 8 + 2 * tq + (e & 1))
                                      : 0.f;
    auto zero4 = [&](float (&F)[4][4]) {
#pragma unroll
        for (int nj = 0; nj < 4; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e) F[nj][e] = 0.f;
    };
    // this warp's [16 rows][32 columns] of a [64][64] tile, fp32 fragments, into two bf16 tiles
    auto store_parts = [&](const float (&F)[4][4], int off_hi, int off_lo) {
#pragma unroll
        for (int nj = 0; nj < 4; ++nj)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = wr * 16 + g + 8 * h, col = (4 * hf + nj) * 8 + 2 * tq;
                const uint32_t off = swz<C::VRB>(row, col >> 3) + (col & 7) * 2;
                uint32_t hi, lo;
                split_bf16x2(make_float2(F[nj][2 * h], F[nj][2 * h + 1]), hi, lo);
                *reinterpret_cast<uint32_t *>(smem + off_hi + off) = hi;
                *reinterpret_cast<uint32_t *>(smem + off_lo + off) = lo;
            }
    };
    auto read_parts = [&](int off_hi, int off_lo, int row, int col) {
        const uint32_t off = swz<C::VRB>(row, col >> 3) + (col & 7) * 2;
        const float2 h = unpack_bf16(*reinterpret_cast<const uint32_t *>(smem + off_hi + off));
        const float2 l = unpack_bf16(*reinterpret_cast<const uint32_t *>(smem + off_lo + off));
        return make_float2(h.x + l.x, h.y + l.y);
    };
    auto bf_v = [&](int off, int row, int col) {  // a bf16 pair of a [64][64] input tile
        return unpack_bf16(*reinterpret_cast<const uint32_t *>(smem + off + swz<C::VRB>(row, col >> 3) + (col & 7) * 2));
    };
    auto bf_q = [&](int row, int col) {  // a bf16 pair of Q
        return unpack_bf16(*reinterpret_cast<const uint32_t *>(sQ + swz<C::QRB>(row, col >> 3) + (col & 7) * 2));
    };
    // F [16 rows][this warp's 32 columns] += A (rows of a row-major tile, KS k-steps) x B, B from
    // rows of a tile [n][k] (NK) or from a tile [k][n] (KN); pp = n-tile pair 2 hf + p2
    auto mma_half_nk = [&](float (&F)[4][4], const uint8_t *at, const uint8_t *bt, auto rb_a, auto rb_b, auto ks) {
        constexpr int RA = decltype(rb_a)::value, RB = decltype(rb_b)::value, KS = decltype(ks)::value;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t a[4];
            lda_rows<RA>(a, at, wr * 16, kk, lane);
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
                uint32_t b[4];
                ldb_nk<RB>(b, bt, 2 * hf + p2, kk, lane);
                mma16816(F[2 * p2], a, b[0], b[1]);
                mma16816(F[2 * p2 + 1], a, b[2], b[3]);
            }
        }
    };
    auto mma_half_kn = [&](float (&F)[4][4], const uint8_t *at, const uint8_t *bt, auto rb_a, auto rb_b, auto ks) {
        constexpr int RA = decltype(rb_a)::value, RB = decltype(rb_b)::value, KS = decltype(ks)::value;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t a[4];
            lda_rows<RA>(a, at, wr * 16, kk, lane);
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
                uint32_t b[4];
                ldb_kn<RB>(b, bt, 2 * hf + p2, kk, lane);
                mma16816(F[2 * p2], a, b[0], b[1]);
                mma16816(F[2 * p2 + 1], a, b[2], b[3]);
            }
        }
    };
    using IQ = std::integral_constant<int, C::QRB>;
    using IV = std::integral_constant<int, C::VRB>;
    using K4 = std::integral_constant<int, 4>;        // k-steps over 64 tokens or 64 value columns
    using KD = std::integral_constant<int, DK / 16>;  // k-steps over the key dimension
    int rr[2];  // this thread's two rows of the chunk
    rr[0] = wr * 16 + g;
    rr[1] = rr[0] + 8;
    auto colof = [&](int nj) { return (4 * hf + nj) * 8 + 2 * tq; };  // first column of a half-tile pair

    load_stage(p.n_chunks - 1);
    cp_async_commit();
    for (int i = p.n_chunks - 1; i >= 0; --i) {
        const long long t0 = (long long)i * kDlTc;
        if (i > 0) prefetch_stage(i - 1);
        // dS' (the adjoint of the state leaving chunk i) as two bf16 parts
#pragma unroll
        for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = s_row(mi, h), col = colof(nj);
                    const uint32_t off = swz<VRB>(row, col >> 3) + (col & 7) * 2;
                    uint32_t hi, lo;
                    split_bf16x2(make_float2(dS[mi][nj][2 * h], dS[mi][nj][2 * h + 1]), hi, lo);
                    *reinterpret_cast<uint32_t *>(smem + C::OFF_GH + off) = hi;
                    *reinterpret_cast<uint32_t *>(smem + C::OFF_GL + off) = lo;
                }
        cp_async_wait<0>();
        __syncthreads();
        // ---- in-chunk log2 decays (warp 0); this thread's share of <S, dS'>
        if (warp == 0) {
            const float v0 = ls[2 * lane] * kDlLog2e;
            const float v1 = v0 + ls[2 * lane + 1] * kDlLog2e;
            float tot = v1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, tot, off);
                if (lane >= off) tot += o;
            }
            const float ex = tot - v1;
            cs[2 * lane] = ex + v0;
            cs[2 * lane + 1] = ex + v1;
        }
        float sd = 0.f;
#pragma unroll
        for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 s = read_parts(C::OFF_SH, C::OFF_SL, s_row(mi, h), colof(nj));
                    sd += s.x * dS[mi][nj][2 * h] + s.y * dS[mi][nj][2 * h + 1];
                }
        __syncthreads();
        const float cL = cs[kDlTc - 1];
        float rt[2] = {0.f, 0.f};   // this warp's row parts of the gradient on c (quad sums)
        float dbr[2] = {0.f, 0.f};  // this warp's parts of dbeta (quad sums)
        float esum = 0.f;           // sum of e over this thread's rows (counted once per quad)

        // ---- E = strictly lower (2^(c_r - c_s) k_r . k_s), fp32, and (I + A)^-1 (A = diag(beta) E)
        // as two bf16 parts arrived with the chunk's inputs;
        // every warp forms K S, Yv = V - diag(gamma) K S and X = diag(beta) Yv for its part
        float Yv[4][4];
        {
            zero4(Yv);
            mma_half_kn(Yv, sK, smem + C::OFF_SH, IQ{}, IV{}, KD{});
            mma_half_kn(Yv, sK, smem + C::OFF_SL, IQ{}, IV{}, KD{});
            float X[4][4];
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = rr[h];
                    const float2 vv = bf_v(C::OFF_V, r, colof(nj));
                    const float gm = ex2(cs[r]), bt = bs[r];
                    Yv[nj][2 * h] = vv.x - gm * Yv[nj][2 * h];
                    Yv[nj][2 * h + 1] = vv.y - gm * Yv[nj][2 * h + 1];
                    X[nj][2 * h] = bt * Yv[nj][2 * h];
                    X[nj][2 * h + 1] = bt * Yv[nj][2 * h + 1];
                }
            store_parts(X, C::OFF_XH, C::OFF_XL);
        }
        __syncthreads();
        // ---- U = (I + A)^-1 X (three products); U and diag(w) U as bf16 parts
        {
            float U[4][4];
            zero4(U);
            mma_half_kn(U, smem + C::OFF_TH, smem + C::OFF_XH, IV{}, IV{}, K4{});
            mma_half_kn(U, smem + C::OFF_TH, smem + C::OFF_XL, IV{}, IV{}, K4{});
            mma_half_kn(U, smem + C::OFF_TL, smem + C::OFF_XH, IV{}, IV{}, K4{});
            store_parts(U, C::OFF_UH, C::OFF_UL);
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float w = ex2(cL - cs[rr[h]]);
                    U[nj][2 * h] *= w;
                    U[nj][2 * h + 1] *= w;
                }
            store_parts(U, C::OFF_WH, C::OFF_WL);
        }
        __syncthreads();
        // ---- dU = P^T dO + diag(w) K dS' (this warp's column half); e_s = w_s (K dS')_s . U_s
        {
            float D[4][4];
            zero4(D);
            mma_half_kn(D, sK, smem + C::OFF_GH, IQ{}, IV{}, KD{});
            mma_half_kn(D, sK, smem + C::OFF_GL, IQ{}, IV{}, KD{});
            float eu[2] = {0.f, 0.f};
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 u = read_parts(C::OFF_UH, C::OFF_UL, rr[h], colof(nj));
                    eu[h] += D[nj][2 * h] * u.x + D[nj][2 * h + 1] * u.y;
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float w = ex2(cL - cs[rr[h]]);
                const float e = w * quad_sum(eu[h]);
                rt[h] -= e;
                esum += (tq == 0) ? e : 0.f;
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    D[nj][2 * h] *= w;
                    D[nj][2 * h + 1] *= w;
                }
            }
            // P^T for this warp's rows s, all 64 columns r: (K Q^T)_sr 2^(c_r - c_s), r >= s
            uint32_t ph[4][4], pl[4][4];
            {
                float Pt[8][4];
#pragma unroll
                for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                    for (int e = 0; e < 4; ++e) Pt[nj][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KQ; ++kk) {
                    uint32_t a[4];
                    lda_rows<QRB>(a, sK, wr * 16, kk, lane);
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        uint32_t b[4];
                        ldb_nk<QRB>(b, sQ, pp, kk, lane);
                        mma_pair(Pt, pp, a, b);
                    }
                }
#pragma unroll
                for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int s = rr[h], r0 = nj * 8 + 2 * tq;
                        const float x0 = (r0 >= s) ? Pt[nj][2 * h] * ex2(cs[r0] - cs[s]) : 0.f;
                        const float x1 = (r0 + 1 >= s) ? Pt[nj][2 * h + 1] * ex2(cs[r0 + 1] - cs[s]) : 0.f;
                        split_bf16x2(make_float2(x0, x1), ph[nj >> 1][(nj & 1) * 2 + h], pl[nj >> 1][(nj & 1) * 2 + h]);
                    }
            }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt)
#pragma unroll
                for (int p2 = 0; p2 < 2; ++p2) {
                    uint32_t b[4];
                    ldb_kn<VRB>(b, sdO, 2 * hf + p2, kt, lane);
                    mma16816(D[2 * p2], ph[kt], b[0], b[1]);
                    mma16816(D[2 * p2 + 1], ph[kt], b[2], b[3]);
                    mma16816(D[2 * p2], pl[kt], b[0], b[1]);
                    mma16816(D[2 * p2 + 1], pl[kt], b[2], b[3]);
                }
            store_parts(D, C::OFF_XH, C::OFF_XL);  // X is dead: every warp has formed U
        }
        __syncthreads();
        // ---- dX = (I + A)^-T dU (this warp's column half); dV; the dots with Yv and V;
        // Zk = -diag(beta gamma) dX
        float dXf[4][4];
        {
            zero4(dXf);
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                uint32_t th[4], tl[4];
                lda_trans<VRB>(th, smem + C::OFF_TH, wr, kt, lane);
                lda_trans<VRB>(tl, smem + C::OFF_TL, wr, kt, lane);
#pragma unroll
                for (int p2 = 0; p2 < 2; ++p2) {
                    uint32_t dh[4], dl[4];
                    ldb_kn<VRB>(dh, smem + C::OFF_XH, 2 * hf + p2, kt, lane);
                    ldb_kn<VRB>(dl, smem + C::OFF_XL, 2 * hf + p2, kt, lane);
                    mma_pair(dXf, p2, th, dh);
                    mma_pair(dXf, p2, th, dl);
                    mma_pair(dXf, p2, tl, dh);
                }
            }
            float ydx[2] = {0.f, 0.f}, vdx[2] = {0.f, 0.f};
            float Z[4][4];
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = rr[h], col = colof(nj);
                    const long long t = t0 + r;
                    const float bt = bs[r];
                    const float f0 = dXf[nj][2 * h], f1 = dXf[nj][2 * h + 1];
                    if (t < p.T)
                        *reinterpret_cast<float2 *>(p.dv + (tok0 + t) * p.DV + zb * 64 + col) =
                            make_float2(bt * f0, bt * f1);
                    const float2 vv = bf_v(C::OFF_V, r, col);
                    ydx[h] += Yv[nj][2 * h] * f0 + Yv[nj][2 * h + 1] * f1;
                    vdx[h] += vv.x * f0 + vv.y * f1;
                    const float m = -bt * ex2(cs[r]);
                    Z[nj][2 * h] = m * f0;
                    Z[nj][2 * h + 1] = m * f1;
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float y = quad_sum(ydx[h]), vx = quad_sum(vdx[h]);
                rt[h] -= bs[rr[h]] * (vx - y);
                dbr[h] += y;
            }
            store_parts(Z, C::OFF_ZH, C::OFF_ZL);
        }
        __syncthreads();  // every warp has read (I + A)^-1 and dU
        store_parts(dXf, C::OFF_TH, C::OFF_TL);  // dX, where (I + A)^-1 was
        __syncthreads();
        // ---- dA = -dX U^T (s < r) and dP = dO U^T (s <= r) with P = (Q K^T) . D, for this warp's
        // column half s: dbeta, the gradient on c, F = diag(beta) dA . D, G1 = dP . D
        float colacc[4][2];
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) colacc[nj][0] = colacc[nj][1] = 0.f;
        float Fm[4][4], G1[4][4];
        {
            float rowm[2] = {0.f, 0.f}, dba[2] = {0.f, 0.f};
            zero4(Fm);
            mma_half_nk(Fm, smem + C::OFF_TH, smem + C::OFF_UH, IV{}, IV{}, K4{});
            mma_half_nk(Fm, smem + C::OFF_TH, smem + C::OFF_UL, IV{}, IV{}, K4{});
            mma_half_nk(Fm, smem + C::OFF_TL, smem + C::OFF_UH, IV{}, IV{}, K4{});
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = rr[e >> 1], s = colof(nj) + (e & 1);
                    if (s < r) {
                        const float Ers = Em[r * kAS + s];
                        const float dA = -Fm[nj][e], bt = bs[r];
                        dba[e >> 1] += dA * Ers;
                        const float m2 = dA * bt * Ers;
                        rowm[e >> 1] += m2;
                        colacc[nj][e & 1] += m2;
                        Fm[nj][e] = bt * dA * ex2(cs[r] - cs[s]);
                    } else {
                        Fm[nj][e] = 0.f;
                    }
                }
            zero4(G1);
            mma_half_nk(G1, sdO, smem + C::OFF_UH, IV{}, IV{}, K4{});
            mma_half_nk(G1, sdO, smem + C::OFF_UL, IV{}, IV{}, K4{});
            float P[4][4];
            zero4(P);
            mma_half_nk(P, sQ, sK, IQ{}, IQ{}, KD{});
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = rr[e >> 1], s = colof(nj) + (e & 1);
                    if (s <= r) {
                        const float d = ex2(cs[r] - cs[s]);
                        const float m1 = G1[nj][e] * P[nj][e] * d;
                        rowm[e >> 1] += m1;
                        colacc[nj][e & 1] += m1;
                        G1[nj][e] *= d;
                    } else {
                        G1[nj][e] = 0.f;
                    }
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                rt[h] += quad_sum(rowm[h]);
                dbr[h] += quad_sum(dba[h]);
            }
        }
        __syncthreads();  // every warp has read E, dX and dU
        store_parts(Fm, C::OFF_FH, C::OFF_FL);  // F, where E was
        store_parts(G1, C::OFF_XH, C::OFF_XL);  // dP . D, where dU was
        {
            float Zq[4][4];  // diag(gamma) dO, where dX was
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 vv = bf_v(C::OFF_DO, rr[h], colof(nj));
                    const float gm = ex2(cs[rr[h]]);
                    Zq[nj][2 * h] = gm * vv.x;
                    Zq[nj][2 * h + 1] = gm * vv.y;
                }
            store_parts(Zq, C::OFF_TH, C::OFF_TL);
        }
        // column parts of the gradient on c (this warp's 32 columns), the last position's extra
#pragma unroll
        for (int nj = 0; nj < 4; ++nj)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float x = colacc[nj][c];
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                x += __shfl_xor_sync(0xffffffffu, x, 8);
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                if (g == 0) colp[warp * kDlTc + colof(nj) + c] = x;
            }
        {
            float ex = esum + ex2(cL) * sd;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ex += __shfl_xor_sync(0xffffffffu, ex, off);
            if (lane == 0) red[warp] = ex;
        }
        __syncthreads();  // F, G1, Zq in shared memory
        // ---- dQ = G1 K + diag(gamma) dO S^T (this warp's half of the DK columns), and
        // gamma_r q_r . (dO S^T)_r
        {
            float Acc[NQ2][4];
#pragma unroll
            for (int j = 0; j < NQ2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) Acc[j][e] = 0.f;
            constexpr int PP = DK / 32;  // n-tile pairs of a half
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                uint32_t a[4];
                lda_rows<VRB>(a, sdO, wr * 16, kt, lane);
#pragma unroll
                for (int p2 = 0; p2 < PP; ++p2) {
                    uint32_t sh[4], sl[4];
                    ldb_nk<VRB>(sh, smem + C::OFF_SH, hf * PP + p2, kt, lane);
                    ldb_nk<VRB>(sl, smem + C::OFF_SL, hf * PP + p2, kt, lane);
                    mma_pair(Acc, p2, a, sh);
                    mma_pair(Acc, p2, a, sl);
                }
            }
            float qd[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < NQ2; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 qq = bf_q(rr[h], (hf * NQ2 + j) * 8 + 2 * tq);
                    qd[h] += qq.x * Acc[j][2 * h] + qq.y * Acc[j][2 * h + 1];
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float gm = ex2(cs[rr[h]]);
                rt[h] += gm * quad_sum(qd[h]);
#pragma unroll
                for (int j = 0; j < NQ2; ++j) {
                    Acc[j][2 * h] *= gm;
                    Acc[j][2 * h + 1] *= gm;
                }
            }
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
                uint32_t ah[4], al[4];
                lda_rows<VRB>(ah, smem + C::OFF_XH, wr * 16, kt, lane);
                lda_rows<VRB>(al, smem + C::OFF_XL, wr * 16, kt, lane);
#pragma unroll
                for (int p2 = 0; p2 < PP; ++p2) {
                    uint32_t b[4];
                    ldb_kn<QRB>(b, sK, hf * PP + p2, kt, lane);
                    mma_pair(Acc, p2, ah, b);
                    mma_pair(Acc, p2, al, b);
                }
            }
#pragma unroll
            for (int j = 0; j < NQ2; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long t = t0 + rr[h];
                    if (t < p.T)
                        *reinterpret_cast<float2 *>(dq_out + (size_t)t * DK + (hf * NQ2 + j) * 8 + 2 * tq) =
                            make_float2(Acc[j][2 * h], Acc[j][2 * h + 1]);
                }
        }
        if (tq == 0) {
            rowp[hf * kDlTc + rr[0]] = rt[0];
            rowp[hf * kDlTc + rr[1]] = rt[1];
            dbs[hf * kDlTc + rr[0]] = dbr[0];
            dbs[hf * kDlTc + rr[1]] = dbr[1];
        }
        // ---- dK = G1^T Q + (F^T + F) K + diag(w) U dS'^T + Zk S^T (this warp's half of DK)
        {
            float Acc[NQ2][4];
#pragma unroll
            for (int j = 0; j < NQ2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) Acc[j][e] = 0.f;
            constexpr int PP = DK / 32;
#pragma unroll 1
            for (int kt = 0; kt < 4; ++kt) {  // k over the chunk's tokens
                uint32_t gh[4], gl[4], fth[4], ftl[4], fh[4], fl[4];
                lda_trans<VRB>(gh, smem + C::OFF_XH, wr, kt, lane);
                lda_trans<VRB>(gl, smem + C::OFF_XL, wr, kt, lane);
                lda_trans<VRB>(fth, smem + C::OFF_FH, wr, kt, lane);
                lda_trans<VRB>(ftl, smem + C::OFF_FL, wr, kt, lane);
                lda_rows<VRB>(fh, smem + C::OFF_FH, wr * 16, kt, lane);
                lda_rows<VRB>(fl, smem + C::OFF_FL, wr * 16, kt, lane);
#pragma unroll
                for (int p2 = 0; p2 < PP; ++p2) {
                    uint32_t bq[4], bk[4];
                    ldb_kn<QRB>(bq, sQ, hf * PP + p2, kt, lane);
                    ldb_kn<QRB>(bk, sK, hf * PP + p2, kt, lane);
                    mma_pair(Acc, p2, gh, bq);
                    mma_pair(Acc, p2, gl, bq);
                    mma_pair(Acc, p2, fth, bk);
                    mma_pair(Acc, p2, ftl, bk);
                    mma_pair(Acc, p2, fh, bk);
                    mma_pair(Acc, p2, fl, bk);
                }
            }
#pragma unroll 1
            for (int kt = 0; kt < 4; ++kt) {  // k over the 64 value columns
                uint32_t wh[4], wl[4], zh[4], zl[4];
                lda_rows<VRB>(wh, smem + C::OFF_WH, wr * 16, kt, lane);
                lda_rows<VRB>(wl, smem + C::OFF_WL, wr * 16, kt, lane);
                lda_rows<VRB>(zh, smem + C::OFF_ZH, wr * 16, kt, lane);
                lda_rows<VRB>(zl, smem + C::OFF_ZL, wr * 16, kt, lane);
#pragma unroll
                for (int p2 = 0; p2 < PP; ++p2) {
                    uint32_t b1[4], b2[4];
                    ldb_nk<VRB>(b1, smem + C::OFF_GH, hf * PP + p2, kt, lane);
                    ldb_nk<VRB>(b2, smem + C::OFF_GL, hf * PP + p2, kt, lane);
                    mma_pair(Acc, p2, wh, b1);
                    mma_pair(Acc, p2, wh, b2);
                    mma_pair(Acc, p2, wl, b1);
                    ldb_nk<VRB>(b1, smem + C::OFF_SH, hf * PP + p2, kt, lane);
                    ldb_nk<VRB>(b2, smem + C::OFF_SL, hf * PP + p2, kt, lane);
                    mma_pair(Acc, p2, zh, b1);
                    mma_pair(Acc, p2, zh, b2);
                    mma_pair(Acc, p2, zl, b1);
                }
            }
#pragma unroll
            for (int j = 0; j < NQ2; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long t = t0 + rr[h];
                    if (t < p.T)
                        *reinterpret_cast<float2 *>(dk_out + (size_t)t * DK + (hf * NQ2 + j) * 8 + 2 * tq) =
                            make_float2(Acc[j][2 * h], Acc[j][2 * h + 1]);
                }
        }
        // ---- dS = gamma_L dS' + Q^T Zq + K^T Zk   (two products each; this warp's part)
        {
            const float gL = ex2(cL);
#pragma unroll
            for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
                for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dS[mi][nj][e] *= gL;
#pragma unroll 1
            for (int kt = 0; kt < 4; ++kt)
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const uint8_t *zt_h = smem + (which ? C::OFF_ZH : C::OFF_TH);
                    const uint8_t *zt_l = smem + (which ? C::OFF_ZL : C::OFF_TL);
                    const uint8_t *yt = which ? sK : sQ;
                    uint32_t b[2][4], bl[2][4];
#pragma unroll
                    for (int p2 = 0; p2 < 2; ++p2) {
                        ldb_kn<VRB>(b[p2], zt_h, 2 * hf + p2, kt, lane);
                        ldb_kn<VRB>(bl[p2], zt_l, 2 * hf + p2, kt, lane);
                    }
#pragma unroll
                    for (int mi = 0; mi < S_MT; ++mi) {
                        uint32_t a[4];
                        lda_trans<QRB>(a, yt, wr * S_MT + mi, kt, lane);
#pragma unroll
                        for (int p2 = 0; p2 < 2; ++p2) {
                            mma_pair(dS[mi], p2, a, b[p2]);
                            mma_pair(dS[mi], p2, a, bl[p2]);
                        }
                    }
                }
        }
        __syncthreads();  // row parts, column parts, dbeta
        // ---- the gradient on c -> suffix sums in the chunk -> dlog_a; dbeta (warp 0, two rows a lane)
        if (warp == 0) {
            float extra = 0.f;
#pragma unroll
            for (int w = 0; w < kDlBwdThreads / 32; ++w) extra += red[w];
            float d[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                float cp = 0.f;  // the four warps of column r's half
#pragma unroll
                for (int w = 0; w < 4; ++w) cp += colp[(4 * (r >> 5) + w) * kDlTc + r];
                d[u] = (rowp[r] + rowp[kDlTc + r]) - cp;
            }
            if (lane == 31) d[1] += extra;
            float tot = d[0] + d[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_down_sync(0xffffffffu, tot, off);
                if (lane + off < 32) tot += o;
            }
            const int r0 = 2 * lane;
            const long long ta = t0 + r0;
            if (ta < p.T) {
                dl_out[ta] = tot;
                db_out[ta] = dbs[r0] + dbs[kDlTc + r0];
            }
            if (ta + 1 < p.T) {
                dl_out[ta + 1] = tot - d[0];
                db_out[ta + 1] = dbs[r0 + 1] + dbs[kDlTc + r0 + 1];
            }
        }
        __syncthreads();  // before the next chunk's loads overwrite shared memory
        if (i > 0) load_stage(i - 1);
        cp_async_commit();
    }
    cp_async_wait<0>();
    if (p.dS0 != nullptr) {
#pragma unroll
        for (int mi = 0; mi < S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<float2 *>(p.dS0 + ((size_t)bh * DK + s_row(mi, h)) * p.DV + zb * 64 +
                                                colof(nj)) = make_float2(dS[mi][nj][2 * h], dS[mi][nj][2 * h + 1]);
    }
}

// dq, dk, dlog_a, dbeta += the partials of the value-column blocks 1..nzb-1, in block order.
__global__ void delta_bwd_reduce_kernel(float *dq, float *dk, float *dl, float *db, const float *part,
                                        long long part_stride, long long ntok, int dim_k, int nparts) {
    const long long nqk = ntok * dim_k;  // even: dim_k is a multiple of 64
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (long long i = i0; i < nqk; i += stride) {  // the stacked [dq | dk], two floats per step
        const long long e = 2 * i;
        float *dst = e < nqk ? dq + e : dk + (e - nqk);
        float2 s = *reinterpret_cast<const float2 *>(dst);
        for (int z = 0; z < nparts; ++z) {
            const float2 x = __ldcs(reinterpret_cast<const float2 *>(part + z * part_stride + e));
            s.x += x.x;
            s.y += x.y;
        }
        *reinterpret_cast<float2 *>(dst) = s;
    }
    for (long long i = i0; i < 2 * ntok; i += stride) {  // dlog_a and dbeta
        float *dst = i < ntok ? dl + i : db + (i - ntok);
        float s = *dst;
        for (int z = 0; z < nparts; ++z) s += __ldcs(part + z * part_stride + 2 * nqk + i);
        *dst = s;
    }
}

template <int DK>
int launch_delta_bwd(const DeltaBwdArgs &a, cudaStream_t s, unsigned int grid) {
    using C = DeltaBwdCfg<DK>;
    static std::atomic<unsigned long long> smem_set{0};
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(delta_bwd_kernel<DK>), C::SMEM);
    if (st) return st;
    delta_bwd_kernel<DK><<<grid, kDlBwdThreads, C::SMEM, s>>>(a);
    return check_launch("delta_bwd_kernel");
}

// Bytes of the states the backward works from (the state entering every chunk), 16-aligned.
size_t delta_states_bytes(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv) {
    return align_up(sizeof(float) * (size_t)(B * H) * (size_t)((T + kDlTc - 1) / kDlTc) * (size_t)dk * (size_t)dv, 16);
}

// Bytes of the chunks' precomputed (I + A)^-1 parts (16 KB a chunk).
size_t delta_wy_bytes(int64_t B, int64_t H, int64_t T) {
    return (size_t)B * (size_t)H * (size_t)((T + kDlTc - 1) / kDlTc) * (2 * kDlTc * 128);
}
// Bytes of the chunks' E, fp32 [64][64] (16 KB a chunk).
size_t delta_e_bytes(int64_t B, int64_t H, int64_t T) {
    return (size_t)B * (size_t)H * (size_t)((T + kDlTc - 1) / kDlTc) * (kDlTc * kDlTc * 4);
}

// Workspace of the backward: the header, the state entering every chunk, every chunk's (I + A)^-1
// parts, and the partials of the value-column blocks after the first (with a checkpoint, which
// holds the states and the inverses, only the header and the partials).  0 when the shape is
// unsupported or the size overflows.
size_t delta_bwd_ws_bytes(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv) {
    const double BH = (double)B * H, nc = (double)((T + kDlTc - 1) / kDlTc);
    const double states = BH * nc * dk * dv * 4.0;
    const double wy = BH * nc * (2.0 * kDlTc * 128 + kDlTc * kDlTc * 4.0);  // inverse parts and E
    const double parts = (double)(dv / 64 - 1) * BH * T * (2.0 * dk + 2.0) * 4.0;
    const double total = sizeof(WsHeader) + states + 16.0 + wy + parts;
    if (total > 9.0e18) return 0;
    return sizeof(WsHeader) + align_up((size_t)states, 16) + (size_t)wy + (size_t)parts;
}

bool delta_supported(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int chunk) {
    return B >= 0 && H >= 0 && T >= 0 && (dk == 64 || dk == 128) && dv > 0 && dv % 64 == 0 && dv <= 1024 &&
           chunk == kDlTc && product_below({B, H}, 16777217.0) && T <= (1ll << 34) &&
           product_below({B, H, T}, 1099511627777.0) && product_below({B, H, dv / 64}, 2147483648.0);
}

}  // namespace
}  // namespace cla

using namespace cla;

extern "C" size_t cla_delta_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                           int chunk) {
    if (!delta_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    return sizeof(WsHeader) + delta_wy_bytes(B, H, T);
}

namespace {
int delta_fwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                   const float *beta, const float *S0, float *o, float *ST, float *ckpt, int64_t B, int64_t H,
                   int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    if (B < 0 || H < 0 || T < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!delta_supported(B, H, T, dim_k, dim_v, chunk))
        return fail(CLA_ERR_UNSUPPORTED, "%s: needs dim_k 64 or 128, dim_v a multiple of 64 up to 1024 and chunk 64 "
                    "(got dim_k %lld, dim_v %lld, chunk %d)", fn, (long long)dim_k, (long long)dim_v, chunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t BH = B * H;
    if (BH == 0) return CLA_OK;
    if (T == 0) {
        if (ST) {
            const size_t sbytes = sizeof(float) * BH * dim_k * dim_v;
            if (S0) CLA_CUDA_TRY(cudaMemcpyAsync(ST, S0, sbytes, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(ST, 0, sbytes, s), fn);
        }
        return CLA_OK;
    }
    if (!q || !k || !v || !log_decay || !beta || !o)
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, log_decay, beta, o required", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v must be 16-byte aligned", fn);
    if (!aligned_or_null({o}, 8) || !aligned_or_null({log_decay, beta, S0, ST}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: o must be 8-byte aligned, log_decay, beta, S0, ST 4-byte", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    if (ws_bytes < sizeof(WsHeader))
        return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, sizeof(WsHeader));
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(WsHeader), s), fn);
    // with room for them (the size query's workspace), the chunks' (I + A)^-1 are formed first, all
    // chunks in parallel; with a header-only workspace the chunk loop forms them itself
    // (a checkpoint holds them after the states, for the backward to reuse)
    const size_t wy_bytes = delta_wy_bytes(B, H, T);
    uint8_t *wy = ckpt != nullptr ? reinterpret_cast<uint8_t *>(ckpt) + delta_states_bytes(B, H, T, dim_k, dim_v)
                  : ws_bytes >= sizeof(WsHeader) + wy_bytes ? static_cast<uint8_t *>(ws) + sizeof(WsHeader)
                                                            : nullptr;
    // with a checkpoint the backward's E too (after the inverse parts)
    float *E = ckpt != nullptr ? reinterpret_cast<float *>(wy + wy_bytes) : nullptr;
    DeltaArgs a;
    memset(&a, 0, sizeof(a));
    a.q = reinterpret_cast<const bf16 *>(q);
    a.k = reinterpret_cast<const bf16 *>(k);
    a.v = reinterpret_cast<const bf16 *>(v);
    a.g = log_decay;
    a.beta = beta;
    a.S0 = S0;
    a.o = o;
    a.ST = ST;
    a.BH = (int)BH;
    a.DV = (int)dim_v;
    a.nzb = (int)(dim_v / 64);
    a.n_chunks = (int)((T + kDlTc - 1) / kDlTc);
    a.T = T;
    a.hdr = static_cast<WsHeader *>(ws);
    a.states = ckpt;
    a.wy = wy;
    a.E = E;
    if (wy != nullptr) {
        const int st = dim_k == 64 ? launch_delta_wy<64>(a, s) : launch_delta_wy<128>(a, s);
        if (st) return st;
    }
    const unsigned int grid = (unsigned int)(BH * (dim_v / 64));
    return dim_k == 64 ? launch_delta_fwd<64>(a, s, grid) : launch_delta_fwd<128>(a, s, grid);
}
}  // namespace

extern "C" size_t cla_delta_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk) {
    if (!delta_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    const double nc = (double)((T + kDlTc - 1) / kDlTc);
    const double bytes = (double)B * H * nc * (dim_k * dim_v * 4.0 + 2.0 * kDlTc * 128 + kDlTc * kDlTc * 4.0) + 16.0;
    return bytes > 9.0e18 ? 0
                          : delta_states_bytes(B, H, T, dim_k, dim_v) + delta_wy_bytes(B, H, T) + delta_e_bytes(B, H, T);
}

extern "C" int cla_delta_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                             const float *beta, const float *S0, float *o, float *ST, int64_t B, int64_t H,
                             int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                             void *stream) {
    return delta_fwd_impl("cla_delta_fwd", q, k, v, log_decay, beta, S0, o, ST, nullptr, B, H, T, dim_k, dim_v,
                          chunk, ws, ws_bytes, stream);
}

extern "C" int cla_delta_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                  const float *beta, const float *S0, float *o, float *ST, float *ckpt, int64_t B,
                                  int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                                  size_t ws_bytes, void *stream) {
    if (ckpt != nullptr && !aligned16(ckpt))
        return fail(CLA_ERR_INVALID_ARG, "cla_delta_fwd_ckpt: ckpt must be 16-byte aligned");
    return delta_fwd_impl("cla_delta_fwd_ckpt", q, k, v, log_decay, beta, S0, o, ST, ckpt, B, H, T, dim_k, dim_v,
                          chunk, ws, ws_bytes, stream);
}

extern "C" size_t cla_delta_bwd_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                               int chunk) {
    if (!delta_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    return delta_bwd_ws_bytes(B, H, T, dim_k, dim_v);
}

namespace {
int delta_bwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                   const float *beta, const float *S0, const uint16_t *dO, const float *dST, float *dq, float *dk,
                   float *dv, float *dlog_decay, float *dbeta, float *dS0, const float *ckpt, int64_t B, int64_t H,
                   int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    if (B < 0 || H < 0 || T < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!delta_supported(B, H, T, dim_k, dim_v, chunk))
        return fail(CLA_ERR_UNSUPPORTED, "%s: needs dim_k 64 or 128, dim_v a multiple of 64 up to 1024 and chunk 64 "
                    "(got dim_k %lld, dim_v %lld, chunk %d)", fn, (long long)dim_k, (long long)dim_v, chunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t BH = B * H;
    if (BH == 0) return CLA_OK;
    if (T == 0) {  // nothing but the final state's adjoint passes through
        if (dS0) {
            const size_t sbytes = sizeof(float) * BH * dim_k * dim_v;
            if (dST) CLA_CUDA_TRY(cudaMemcpyAsync(dS0, dST, sbytes, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(dS0, 0, sbytes, s), fn);
        }
        return CLA_OK;
    }
    if (!q || !k || !v || !log_decay || !beta || !dO || !dq || !dk || !dv || !dlog_decay || !dbeta)
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, log_decay, beta, dO, dq, dk, dv, dlog_decay, dbeta required",
                    fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, dO must be 16-byte aligned", fn);
    if (!aligned_or_null({dq, dk, dv, dS0, dST, S0}, 8) || !aligned_or_null({log_decay, beta, dlog_decay, dbeta}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: dq, dk, dv, dS0, dST, S0 must be 8-byte aligned, log_decay, beta, "
                    "dlog_decay, dbeta 4-byte", fn);
    if (ckpt != nullptr && !aligned16(ckpt)) return fail(CLA_ERR_INVALID_ARG, "%s: ckpt must be 16-byte aligned", fn);
    // with a checkpoint the states pass is skipped and the workspace holds the header and the partials only
    const size_t full = delta_bwd_ws_bytes(B, H, T, dim_k, dim_v);
    if (full == 0) return fail(CLA_ERR_UNSUPPORTED, "%s: workspace size overflows", fn);
    const size_t states_b = delta_states_bytes(B, H, T, dim_k, dim_v);
    const size_t wy_b = delta_wy_bytes(B, H, T) + delta_e_bytes(B, H, T);  // inverse parts, then E
    const size_t need = ckpt ? full - states_b - wy_b : full;
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    if (ws_bytes < need) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, need);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(WsHeader), s), fn);
    const int n_chunks = (int)((T + kDlTc - 1) / kDlTc);
    float *ws_states = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + sizeof(WsHeader));
    uint8_t *ws_wy = reinterpret_cast<uint8_t *>(ws_states) + states_b;
    const unsigned int grid = (unsigned int)(BH * (dim_v / 64));
    const float *states = ckpt ? ckpt : ws_states;
    // every chunk's (I + A)^-1: from the checkpoint, else formed here (before the states pass, which
    // uses them too)
    const uint8_t *wy = ckpt ? reinterpret_cast<const uint8_t *>(ckpt) + states_b : ws_wy;
    const float *Ech = reinterpret_cast<const float *>(wy + delta_wy_bytes(B, H, T));
    // the states pass (no checkpoint): the forward kernel writes the state entering every chunk, no output
    if (!ckpt) {
        DeltaArgs f;
        memset(&f, 0, sizeof(f));
        f.q = reinterpret_cast<const bf16 *>(q);
        f.k = reinterpret_cast<const bf16 *>(k);
        f.v = reinterpret_cast<const bf16 *>(v);
        f.g = log_decay;
        f.beta = beta;
        f.S0 = S0;
        f.states = ws_states;
        f.BH = (int)BH;
        f.DV = (int)dim_v;
        f.nzb = (int)(dim_v / 64);
        f.n_chunks = n_chunks;
        f.T = T;
        f.hdr = static_cast<WsHeader *>(ws);
        f.wy = ws_wy;
        f.E = reinterpret_cast<float *>(ws_wy + delta_wy_bytes(B, H, T));
        int st = dim_k == 64 ? launch_delta_wy<64>(f, s) : launch_delta_wy<128>(f, s);
        if (st) return st;
        st = dim_k == 64 ? launch_delta_fwd<64>(f, s, grid) : launch_delta_fwd<128>(f, s, grid);
        if (st) return st;
    }
    DeltaBwdArgs a;
    memset(&a, 0, sizeof(a));
    a.q = reinterpret_cast<const bf16 *>(q);
    a.k = reinterpret_cast<const bf16 *>(k);
    a.v = reinterpret_cast<const bf16 *>(v);
    a.dO = reinterpret_cast<const bf16 *>(dO);
    a.g = log_decay;
    a.beta = beta;
    a.dST = dST;
    a.states = states;
    a.wy = wy;
    a.E = Ech;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dlog = dlog_decay;
    a.dbeta = dbeta;
    a.dS0 = dS0;
    a.part = dim_v > 64 ? reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws_states) + (ckpt ? 0 : states_b + wy_b))
                        : nullptr;
    a.part_stride = (long long)BH * T * (2 * dim_k + 2);
    a.BH = (int)BH;
    a.DV = (int)dim_v;
    a.nzb = (int)(dim_v / 64);
    a.n_chunks = n_chunks;
    a.T = T;
    const int st2 = dim_k == 64 ? launch_delta_bwd<64>(a, s, grid) : launch_delta_bwd<128>(a, s, grid);
    if (st2) return st2;
    if (a.nzb > 1) {
        const long long ntok = (long long)BH * T;
        const long long work = ntok * dim_k;
        const unsigned int blocks = (unsigned int)std::min<long long>((work + 255) / 256, 152LL * 16);
        delta_bwd_reduce_kernel<<<blocks, 256, 0, s>>>(dq, dk, dlog_decay, dbeta, a.part, a.part_stride, ntok,
                                                       (int)dim_k, a.nzb - 1);
        return check_launch("delta_bwd_reduce_kernel");
    }
    return CLA_OK;
}
}  // namespace

extern "C" int cla_delta_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                             const float *beta, const float *S0, const uint16_t *dO, const float *dST, float *dq,
                             float *dk, float *dv, float *dlog_decay, float *dbeta, float *dS0, int64_t B,
                             int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                             size_t ws_bytes, void *stream) {
    return delta_bwd_impl("cla_delta_bwd", q, k, v, log_decay, beta, S0, dO, dST, dq, dk, dv, dlog_decay, dbeta, dS0,
                          nullptr, B, H, T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}

extern "C" int cla_delta_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                  const float *beta, const float *S0, const uint16_t *dO, const float *dST, float *dq,
                                  float *dk, float *dv, float *dlog_decay, float *dbeta, float *dS0,
                                  const float *ckpt, int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                  int chunk, void *ws, size_t ws_bytes, void *stream) {
    return delta_bwd_impl("cla_delta_bwd_ckpt", q, k, v, log_decay, beta, S0, dO, dST, dq, dk, dv, dlog_decay, dbeta,
                          dS0, ckpt, B, H, T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}
