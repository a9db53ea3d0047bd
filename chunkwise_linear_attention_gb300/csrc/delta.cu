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
#include "cla_internal.cuh"
#include "mma_sync.cuh"

namespace cla {
namespace {

typedef __nv_bfloat16 bf16;

constexpr float kDlLog2e = 1.4426950408889634f;
constexpr int kDlTc = 64;        // tokens per chunk
constexpr int kDlThreads = 128;  // warp w: rows 16w..16w+15 of a chunk

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
    static constexpr int A_FLOATS = kDlTc * (kDlTc + 1);
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
    float *o, *ST;
    int BH, DV, nzb, n_chunks;
    long long T;
    WsHeader *hdr;
};

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
        cp_async_wait<0>();
        __syncthreads();
        // ---- in-chunk log2 decays (warp 0) and the state's bf16 parts (everyone)
        if (warp == 0) {
            float v0 = ls[2 * lane], v1 = ls[2 * lane + 1];
            const float b0 = bs[2 * lane], b1 = bs[2 * lane + 1];
            if (!isfinite(v0) || !isfinite(v1) || !isfinite(b0) || !isfinite(b1)) atomicOr(&p.hdr->error, kErrRange);
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
        write_state_parts();
        __syncthreads();
        const float cL = cs[kDlTc - 1];

        // ---- A = strictly lower (beta_r 2^(c_r - c_s) k_r . k_s), this warp's 16 rows
        {
            float F[8][4];
            zero8(F);
#pragma unroll 2
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t a[4];
                ldsm_x4(smem_u32(st + C::OFF_K + swz<C::QRB>(arow, 2 * kk + (lane >> 4))), a);
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    uint32_t b[4];
                    const int brow = 16 * pp + (lane & 7) + (lane >> 4) * 8;
                    ldsm_x4(smem_u32(st + C::OFF_K + swz<C::QRB>(brow, 2 * kk + ((lane >> 3) & 1))), b);
                    mma16816(F[2 * pp], a, b[0], b[1]);
                    mma16816(F[2 * pp + 1], a, b[2], b[3]);
                }
            }
#pragma unroll
            for (int nj = 0; nj < 8; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = warp * 16 + g + 8 * (e >> 1), s = nj * 8 + 2 * tq + (e & 1);
                    Am[r * (kDlTc + 1) + s] = (s < r) ? bs[r] * ex2(cs[r] - cs[s]) * F[nj][e] : 0.f;
                }
        }
        __syncthreads();
        // ---- T = (I + A)^-1, unit lower triangular: thread j < 64 builds column j top-down,
        // T[r][j] = -sum_{s<r} A[r][s] T[s][j] (T[s][j] = 0 above row j, 1 on it), in registers,
        // then stores it as two bf16 parts (row r, column j of the [64][64] tiles)
        if (tid < kDlTc) {
            const int j = tid;
            float tc[kDlTc];
#pragma unroll
            for (int r = 0; r < kDlTc; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < r; ++s2) acc = fmaf(Am[r * (kDlTc + 1) + s2], tc[s2], acc);
                tc[r] = (r < j) ? 0.f : (r == j ? 1.f : -acc);
            }
#pragma unroll
            for (int r = 0; r < kDlTc; ++r) {
                const uint32_t off = swz<C::VRB>(r, j >> 3) + (j & 7) * 2;
                const uint32_t bits = __float_as_uint(tc[r]) & 0xffff0000u;
                const float rest = tc[r] - __uint_as_float(bits);  // exact
                *reinterpret_cast<uint16_t *>(smem + C::OFF_TH + off) = (uint16_t)(bits >> 16);
                *reinterpret_cast<uint16_t *>(smem + C::OFF_TL + off) = (uint16_t)(__float_as_uint(rest) >> 16);
            }
        }
        __syncthreads();

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
        {
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
int launch_delta_fwd(const DeltaArgs &a, cudaStream_t s, unsigned int grid) {
    using C = DeltaCfg<DK>;
    static std::atomic<unsigned long long> smem_set{0};
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(delta_fwd_kernel<DK>), C::SMEM);
    if (st) return st;
    delta_fwd_kernel<DK><<<grid, kDlThreads, C::SMEM, s>>>(a);
    return check_launch("delta_fwd_kernel");
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
    return sizeof(WsHeader);
}

extern "C" int cla_delta_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                             const float *beta, const float *S0, float *o, float *ST, int64_t B, int64_t H,
                             int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                             void *stream) {
    clear_error();
    const char *fn = "cla_delta_fwd";
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
    const unsigned int grid = (unsigned int)(BH * (dim_v / 64));
    return dim_k == 64 ? launch_delta_fwd<64>(a, s, grid) : launch_delta_fwd<128>(a, s, grid);
}
