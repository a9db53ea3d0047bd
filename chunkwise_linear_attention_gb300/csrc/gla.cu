// gla.cu -- gated linear attention (one decay per key dimension), forward and
// backward, chunkwise, for GB300 (sm_103a).
//
// "Parallel Scan" (zerotofrontier.app), "What one combine costs" (a diagonal
// transition: one decay per state entry) and "The chunkwise algorithm" (the
// GLA form S_t = G_t (.) S_{t-1} + k_t^T v_t, o_t = q_t S_t), with G_t[i][j] =
// a_t[i]: every key dimension i has its own decay.
//
// With c_t[i] the in-chunk cumulative log2 decay of dimension i up to token t
// (c includes the chunk's first token) and m the chunk's 32nd token, the
// decay between a read at r and a write at s <= r factors through m:
//     2^(c_r - c_s) = 2^(c_r - c_m) * 2^(c_m - c_s)
// so, with Q~ = Q (.) 2^(c - c_m) and K~ = K (.) 2^(c_m - c) (per element),
//     O_chunk = (Q~ K~^T . M) V + Q~ (diag(2^c_m) S_prev)
//     S_next  = diag(2^(c_L - c_m)) (diag(2^c_m) S_prev + K~^T V)
// (M the causal mask, c_L the chunk's last token).  Every factor except the
// operand scalings of Q~ and K~ is at most 1; those two are at most the decay
// over 32 tokens.  The kernel therefore needs |c_t - c_m| <= 120 in every
// dimension of every chunk (a gate product over 32 tokens of at least
// 2^-120) and finite log decays; a chunk outside that range sets an error
// flag that cla_check_status reports (the products would overflow fp32).
//
// Q~, K~ and the state are scaled in fp32 and split into bf16 high and low
// parts, and each product takes the parts that keep the rounding below the
// outputs' tolerance: Q~ K~^T and Q~ S' as hi.hi + hi.lo + lo.hi, P V and
// K~^T V as hi + lo (V is an exact bf16 input).  Every traversal (the
// forward, the backward's reversed dV traversal and its dQ / dK traversals)
// runs its products on tcgen05.mma (kind::f16, fp32 accumulators in tensor
// memory).
//
// Chunk parallelism as in chunk_la.cu: a block owns one segment of chunks of
// one (batch, head) and 64 value columns; phase 1 folds the segment into one
// affine pair (diag(alpha_seg), dS_seg), now with one decay per key
// dimension; decoupled look-back over earlier segments gives the incoming
// state; phase 2 runs the chunks from it and writes O.
#include "cla_internal.cuh"
#include "mma_sync.cuh"
#include "tc_ptx.cuh"

namespace cla {
namespace {

typedef __nv_bfloat16 bf16;

constexpr float kGlaLog2e = 1.4426950408889634f;
constexpr int kGlaTc = 64;        // tokens per chunk
constexpr int kGlaMid = 31;       // reference token of a chunk
constexpr float kGlaSpan = 120.f; // largest |c_t - c_mid| (log2) the operand scalings allow
constexpr int kGlaSegChoices[4] = {64, 32, 16, 8};
constexpr long long kGlaMinBlocks = 1024;

// One traversal of the gated recurrence.  Forward (rev = 0): q, k, v, S0 -> o, ST.  Reversed
// (rev = 1, the adjoint of the backward): token t' of the traversal is token T-1-t' of the
// arrays and its decay is the one of token T-t' (none for t' = 0), which turns the adjoint
// recursion Sbar_t = q_t^T obar_t + diag(a_{t+1}) Sbar_{t+1} into the same forward form; with
// q <- k, k <- q, v <- dO and S0 <- dST it gives o = dV and ST = Sbar_0, and ST is then scaled
// by a_0 to give dS0.
struct GlaArgs {
    const bf16 *q, *k, *v;  // q, k: [BH][T][DK]; v: [BH][T][DV]
    const float *g;         // [BH][T][DK] natural-log decays
    const float *S0;        // [BH][DK][DV] or NULL
    float *o;               // [BH][T][DV]
    float *ST;              // [BH][DK][DV] or NULL
    int rev;
    int BH, DV, nzb, n_chunks, seg_chunks, n_seg;
    long long T;
    WsHeader *hdr;
    unsigned int *flags;  // [unit]
    float *alpha;         // [unit][DK]
    float4 *agg, *incl;   // [unit][tiles][threads]
    float *seg_out;       // [n_seg][BH][DK][DV] or NULL: the state entering each segment, saved
};

// ----------------------------------------------------------------- forward on tcgen05
// One traversal of the gated recurrence on the fifth-generation tensor cores.
// Per 64-token chunk, with Q~ = Q (.) 2^(c - c_m), K~ = K (.) 2^(c_m - c) and
// S' = diag(2^c_m) S (each split into two bf16 parts by the threads):
//     P     = Q~ K~^T                       (M = 64, N = 64, K = DK)   three products
//     O     = Q~ S'                         (M = 64, N = 64, K = DK)   three products
//     U     = K~^T V                        (M = DK, N = 64, K = 64)   two products
//     O    += (P . M)_hi V + (P . M)_lo V   (A from tensor memory)     two products
//     S_next = diag(2^(c_L - c_m)) (S' + U)                            threads
// with fp32 accumulators in tensor memory.  The block's 8 warps prepare the
// operands, mask the scores and apply the state update (warps w and w + 4 read
// lane quarter w & 3 of tensor memory and split its columns); one elected lane
// of warp 0 issues the products, whose completion every thread waits for on an
// mbarrier (bounded waits).  Operand tiles use the 128-byte swizzle: Q~ and K~
// K-major ([64 tokens][DK] in 64-element blocks; K~ is also the MN-major A of
// U), V and S' MN-major.  A warp reads its own quarter of tensor-memory lanes:
// the 64-row accumulators keep row 16q + i in lane 32q + i (i < 16), the DK-row
// one (DK = 128) row r in lane r.
//
// Stages are filled by TMA (one thread issues, completion on a per-stage
// mbarrier; rows past the ends of the arrays read as zeros).  A tile copy keeps
// the array order of rows, so in the reversed traversal (token t' is array token
// T-1-t') row j of a stage holds traversal position 63 - j: the in-chunk sums run
// from the last row up, the midpoint and the chunk's end sit at rows 63 - m and
// 0, and the causal mask keeps the rows at and below the diagonal row.
//
// Segments and look-back as before: phase 1 folds the segment's chunks into
// (diag(alpha_seg), dS_seg) from a zero state, decoupled look-back gives the
// incoming state, phase 2 runs the chunks from it and writes O.
template <int DK>
struct GlaTcCfg {
    static constexpr int KB = DK / 64;             // 64-element blocks along the key dimension
    static constexpr int QT_BYTES = KB * 64 * 128;  // a [64 tokens][DK] bf16 operand tile
    static constexpr int V_BYTES = 64 * 128;        // a [64 tokens][64 columns] bf16 operand tile
    static constexpr int G_BYTES = 64 * DK * 4;     // log decays, then in-chunk cumulative log2 decays
    // one stage: Q (then the high part of Q~), K (then K~'s high part), V, G
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = QT_BYTES;
    static constexpr int OFF_V = 2 * QT_BYTES;
    static constexpr int OFF_G = 2 * QT_BYTES + V_BYTES;
    static constexpr int STAGE = 2 * QT_BYTES + V_BYTES + G_BYTES;
    static constexpr int OFF_QL = 2 * STAGE;            // low part of Q~
    static constexpr int OFF_KL = OFF_QL + QT_BYTES;    // low part of K~
    static constexpr int OFF_SH = OFF_KL + QT_BYTES;    // S' high part, [DK rows][64 columns] MN-major
    static constexpr int OFF_SL = OFF_SH + DK * 128;
    static constexpr int OFF_AS = OFF_SL + DK * 128;    // alpha of the segment per key dimension
    static constexpr int OFF_BAR = OFF_AS + DK * 4;     // four mbarriers: two products, two stage loads
    static constexpr int SMEM = OFF_BAR + 32 + 1024;    // + alignment slack of the 1024-byte base
    static constexpr int MIN_BLOCKS = (2 * (SMEM + 1024) <= 228 * 1024) ? 2 : 1;
    // tensor memory: scores, masked score parts, output, state product
    static constexpr uint32_t C_P = 0, C_PB = 64, C_O = 128, C_U = 192, TMEM_COLS = 256;
    static constexpr int SC = (DK == 128) ? 32 : 16;  // state columns per thread
    static_assert(STAGE % 1024 == 0 && QT_BYTES % 1024 == 0, "1024-byte aligned operand tiles");
    static_assert(2 * QT_BYTES >= 64 * 64 * 4, "the output tile fits over a stage's Q~ and K~");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

constexpr int kGlaTcThreads = 256;

// Tensor maps of a traversal's operands ([BH][T][cols] arrays): q, k and v in
// 128-byte-swizzled boxes of 64 tokens x 64 columns (bf16), log decays in plain boxes of
// 64 tokens x d_k (fp32).  Rows past T read as zeros (log a = 0 for the padding tokens).
struct GlaMaps {
    CUtensorMap q, k, v, g;
};

template <int DK, bool REV>
__global__ void __launch_bounds__(kGlaTcThreads, GlaTcCfg<DK>::MIN_BLOCKS)
    gla_tc_kernel(const GlaArgs p, const __grid_constant__ GlaMaps maps) {
    using C = GlaTcCfg<DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    __shared__ uint32_t s_tmem;
    __shared__ unsigned int s_ticket, s_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t barA = sbase + C::OFF_BAR, barB = barA + 8, barL = barA + 16;  // barL + 8 stage

    // tensor memory first (before taking a ticket, so every ticket holder owns its columns)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 0) {
        mbar_init(barA, 1);
        mbar_init(barB, 1);
        mbar_init(barL, 1);
        mbar_init(barL + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ticket = atomicAdd(&p.hdr->ticket[0], 1u);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int q = warp & 3, hf = warp >> 2;              // lane quarter, column half
    const uint32_t tlane = (uint32_t)(q * 32) << 16;     // this warp's lane quarter
    const unsigned int tk = s_ticket;
    const int per_seg = p.BH * p.nzb;
    const int seg = (int)(tk / per_seg);
    const int bh = (int)(tk % per_seg) / p.nzb;
    const int zb = (int)(tk % per_seg) % p.nzb;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
    const int nc = c_end - c_begin;
    const size_t unit = ((size_t)seg * p.BH + bh) * p.nzb + zb;
    bool timed_out = false;
    uint32_t phA = 0u, phB = 0u;
    auto waitA = [&]() {
        if (!mbar_wait(barA, phA)) timed_out = true;
        phA ^= 1u;
    };
    auto waitB = [&]() {
        if (!mbar_wait(barB, phB)) timed_out = true;
        phB ^= 1u;
    };
    uint32_t phL = 0u;  // bit s: parity of stage s's next load
    auto stage_ready = [&](int stage) {
        if (!mbar_wait(barL + 8u * (uint32_t)stage, (phL >> stage) & 1u)) timed_out = true;
        phL ^= 1u << stage;
    };
    // stage rows of the chunk's midpoint token and of its last token
    constexpr int MID = REV ? kGlaTc - 1 - kGlaMid : kGlaMid;
    constexpr int LAST = REV ? 0 : kGlaTc - 1;

    const float *Gb = p.g + (size_t)bh * p.T * DK;
    float *alpha_s = reinterpret_cast<float *>(smem + C::OFF_AS);

    // array row of a chunk's stage row 0: the chunk's first token, or (reversed) the array
    // token of its last traversal position (negative in a ragged last chunk)
    auto row0_of = [&](int chunk) {
        return REV ? p.T - (long long)kGlaTc * (chunk + 1) : (long long)kGlaTc * chunk;
    };
    // Q, K into their K-major swizzled operand positions, V into its MN-major one, G plain.  The
    // reversed traversal's decay of position t' is array token T - t' (none for t' = 0: the
    // row past the end reads as zero): its G tile starts one row later.
    auto load_stage = [&](int stage, int chunk, bool withQ) {
        if (tid != 0) return;
        const uint32_t bar = barL + 8u * (uint32_t)stage, s0 = smem_u32(smem + stage * C::STAGE);
        mbar_expect_tx(bar, (uint32_t)((withQ ? 2 : 1) * C::QT_BYTES + C::V_BYTES + C::G_BYTES));
        const int y = (int)row0_of(chunk);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(s0 + C::OFF_K + kb * 8192, &maps.k, kb * 64, y, bh, bar);
            if (withQ) tma_load_3d(s0 + C::OFF_Q + kb * 8192, &maps.q, kb * 64, y, bh, bar);
        }
        tma_load_3d(s0 + C::OFF_V, &maps.v, zb * 64, y, bh, bar);
        tma_load_3d(s0 + C::OFF_G, &maps.g, 0, REV ? y + 1 : y, bh, bar);
    };
    // In-chunk cumulative log2 decays, in place (the last DK threads, which issue no products:
    // thread cdim >= 0 scans dimension cdim in traversal order), with the range check; returns
    // (to that thread) the chunk's total c_L[cdim].  Positions past the sequence's end decay by
    // nothing (the reversed traversal's first one past the end would otherwise read a_0's row).
    const int cdim = tid - (kGlaTcThreads - DK);
    auto cumulate = [&](int stage, int chunk) {
        float *G = reinterpret_cast<float *>(smem + stage * C::STAGE + C::OFF_G);
        float total = 0.f;
        if (cdim >= 0) {
            const long long n_tok = p.T - (long long)kGlaTc * chunk;  // positions below are tokens
            float run = 0.f, lo = 0.f, hi = 0.f;
            bool finite = true;
#pragma unroll 8
            for (int t = 0; t < kGlaTc; ++t) {
                const int row = REV ? kGlaTc - 1 - t : t;
                const float l = (REV && t >= n_tok) ? 0.f : G[row * DK + cdim];
                finite = finite && isfinite(l);
                run += l * kGlaLog2e;
                G[row * DK + cdim] = run;
                lo = fminf(lo, run);
                hi = fmaxf(hi, run);
            }
            const float cm = G[MID * DK + cdim];
            // the running sum starts at 0 before token 0: include it in the span as well
            if (!finite || hi - cm > kGlaSpan || cm - lo > kGlaSpan || cm > kGlaSpan)
                atomicOr(&p.hdr->error, kErrRange);
            total = run;
        }
        return total;
    };

    // K~ = K 2^(c_m - c) (high part over K, low part in KL) and, withQ, Q~ = Q 2^(c - c_m).
    auto scale_operands = [&](int stage, bool withQ) {
        uint8_t *st = smem + stage * C::STAGE;
        const float *G = reinterpret_cast<const float *>(st + C::OFF_G);
        constexpr int QC = DK / 8;  // 8-element groups of a row
        static_assert(kGlaTc * QC % kGlaTcThreads == 0 && kGlaTcThreads % QC == 0, "whole rounds, fixed columns");
        // a thread keeps its 8 key dimensions (the same in every round) and steps over rows
        const int c16 = tid % QC;
        float2 nm[4];  // -c_m of the thread's dimensions
        {
            const float4 *cmid = reinterpret_cast<const float4 *>(G + MID * DK + c16 * 8);
            const float4 ma = cmid[0], mb = cmid[1];
            nm[0] = make_float2(-ma.x, -ma.y);
            nm[1] = make_float2(-ma.z, -ma.w);
            nm[2] = make_float2(-mb.x, -mb.y);
            nm[3] = make_float2(-mb.z, -mb.w);
        }
#pragma unroll
        for (int it = 0; it < kGlaTc * QC / kGlaTcThreads; ++it) {
            const int row = tid / QC + it * (kGlaTcThreads / QC);
            const float4 *crow = reinterpret_cast<const float4 *>(G + row * DK + c16 * 8);
            float2 d[4];  // c - c_m
            {
                const float4 a = crow[0], b = crow[1];
                d[0] = __fadd2_rn(make_float2(a.x, a.y), nm[0]);
                d[1] = __fadd2_rn(make_float2(a.z, a.w), nm[1]);
                d[2] = __fadd2_rn(make_float2(b.x, b.y), nm[2]);
                d[3] = __fadd2_rn(make_float2(b.z, b.w), nm[3]);
            }
            const uint32_t off = (uint32_t)((c16 >> 3) * 8192) + sw128(row, (c16 & 7) * 8);
            {
                const uint4 kv = *reinterpret_cast<const uint4 *>(st + C::OFF_K + off);
                const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_bf16x2(__fmul2_rn(unpack_bf16(w[e]), make_float2(ex2(-d[e].x), ex2(-d[e].y))), hi[e], lo[e]);
                *reinterpret_cast<uint4 *>(st + C::OFF_K + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + C::OFF_KL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if (withQ) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(st + C::OFF_Q + off);
                const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_bf16x2(__fmul2_rn(unpack_bf16(w[e]), make_float2(ex2(d[e].x), ex2(d[e].y))), hi[e], lo[e]);
                *reinterpret_cast<uint4 *>(st + C::OFF_Q + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + C::OFF_QL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
    };


    // This thread's state: one row (key dimension) srow and SC consecutive columns of half hf.
    // DK = 128: row 32 q + lane (the lane of a 128-row accumulator), columns 32 hf + {0..31}.
    // DK = 64: row 16 q + (lane & 15), columns 32 hf + 16 (lane >> 4) + {0..15} (the paired-half
    // shape of a 64-row accumulator).
    constexpr int SC = C::SC;
    const int srow = (DK == 128) ? 32 * q + lane : 16 * q + (lane & 15);
    const int scol0 = (DK == 128) ? 32 * hf : 32 * hf + 16 * (lane >> 4);
    auto scol = [&](int j) { return scol0 + j; };
    float S[SC];
    // the state product U of this thread's row, from tensor memory
    auto load_u = [&](float (&u)[SC]) {
        uint32_t r[SC];
        tmem_ld_cols<SC>(tmem + tlane + C::C_U + (uint32_t)(32 * hf), r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < SC; ++j) u[j] = __uint_as_float(r[j]);
    };
    // S' = diag(2^c_m) S in place, and its two bf16 parts into the MN-major B tile [DK][64]
    auto state_to_mid = [&](int stage) {
        const float *G = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_G);
        const float f = ex2(G[MID * DK + srow]);
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] *= f;
    };
    auto write_sb = [&]() {
#pragma unroll
        for (int j8 = 0; j8 < SC / 8; ++j8) {  // 8 consecutive columns per 16-byte store
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(make_float2(S[8 * j8 + 2 * e], S[8 * j8 + 2 * e + 1]), hi[e], lo[e]);
            const uint32_t off = sw128(srow, scol(8 * j8));
            *reinterpret_cast<uint4 *>(smem + C::OFF_SH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(smem + C::OFF_SL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };
    // S_next = diag(2^(c_L - c_m)) (S' + U)
    auto state_finish = [&](int stage) {
        const float *G = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_G);
        const float f = ex2(G[LAST * DK + srow] - G[MID * DK + srow]);
        float u[SC];
        load_u(u);
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] = f * (S[j] + u[j]);
    };

    // ---- descriptors (built once; a K step adds a constant to the start-address field)
    auto qdesc = [&](uint32_t off) { return smem_desc(sbase + off, 16, 1024); };      // K-major
    auto ktdesc = [&](uint32_t off) { return smem_desc(sbase + off, 8192, 1024); };   // MN-major A (K~^T)
    auto mndesc = [&](uint32_t off) { return smem_desc(sbase + off, 8192, 1024); };   // MN-major B
    auto kstep_k = [&](int kk) { return (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4); };  // K-major
    auto kstep_mn = [&](int kk) { return (uint64_t)((kk * 2048) >> 4); };                      // MN-major
    constexpr uint32_t id_s = idesc_bf16(64, 64, 0, 0);   // scores: Q~ K~^T
    constexpr uint32_t id_o = idesc_bf16(64, 64, 0, 1);   // Q~ S', P V
    constexpr uint32_t id_u = idesc_bf16(DK, 64, 1, 1);   // K~^T V
    // U = K~_hi^T V + K~_lo^T V into C_U (stage's K~ and V)
    auto issue_u = [&](int stage) {
        const uint32_t so = (uint32_t)(stage * C::STAGE);
        const uint64_t b0 = mndesc(so + C::OFF_V);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const uint64_t a0 = ktdesc(part ? C::OFF_KL : so + C::OFF_K);
#pragma unroll
            for (int kk = 0; kk < kGlaTc / 16; ++kk)
                mma_ss_w(tmem + C::C_U, a0 + kstep_mn(kk), b0 + kstep_mn(kk), id_u, (part | kk) ? 1u : 0u);
        }
    };
    // P = Q~ K~^T (hi hi, hi lo, lo hi) into C_P and O = Q~ S' (hi hi, hi lo, lo hi) into C_O
    auto issue_p_o = [&](int stage) {
        const uint32_t so = (uint32_t)(stage * C::STAGE);
        const uint64_t qh = qdesc(so + C::OFF_Q), ql = qdesc(C::OFF_QL);
        const uint64_t kh = qdesc(so + C::OFF_K), kl = qdesc(C::OFF_KL);
        const uint64_t sh = mndesc(C::OFF_SH), sl = mndesc(C::OFF_SL);
#pragma unroll
        for (int part = 0; part < 3; ++part) {
            const uint64_t a0 = (part == 2) ? ql : qh;
            const uint64_t bp = (part == 1) ? kl : kh, bs = (part == 1) ? sl : sh;
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                mma_ss_w(tmem + C::C_P, a0 + kstep_k(kk), bp + kstep_k(kk), id_s, (part | kk) ? 1u : 0u);
                mma_ss_w(tmem + C::C_O, a0 + kstep_k(kk), bs + kstep_mn(kk), id_o, (part | kk) ? 1u : 0u);
            }
        }
    };
    // O += (P . M)_hi V + (P . M)_lo V, the masked parts from tensor memory: tokens 16kk.. lie in
    // piece kk / 2, its high part in the piece's columns 0..15, the low part in 16..31
    auto issue_pv = [&](int stage) {
        const uint64_t b0 = mndesc((uint32_t)(stage * C::STAGE) + C::OFF_V);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kk = 0; kk < kGlaTc / 16; ++kk) {
                const uint32_t acol = C::C_PB + (uint32_t)(kk >> 1) * 32 + part * 16 + (kk & 1) * 8;
                mma_ts_w(tmem + C::C_O, tmem + acol, b0 + kstep_mn(kk), id_o, 1u);
            }
    };

    // Causal mask of the scores (stage rows s <= r; reversed, s >= r), split into two bf16 parts as
    // the A operand of P V: row r = 16 q + (lane & 15), the 32-token piece hf; threads 0..15 take
    // tokens s0.., 16..31 tokens s0 + 16..
    auto mask_scores = [&]() {
        const int r = 16 * q + (lane & 15);
        {
            const int s0 = hf * 32;
            uint32_t pr[16];
            tmem_ld16x2(tmem + tlane + C::C_P + (uint32_t)s0, pr);
            tmem_ld_wait();
            const int sb = s0 + 16 * (lane >> 4);
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int s = sb + 2 * j;
                float2 v = make_float2(__uint_as_float(pr[2 * j]), __uint_as_float(pr[2 * j + 1]));
                if (REV ? s < r : s > r) v.x = 0.f;
                if (REV ? s + 1 < r : s + 1 > r) v.y = 0.f;
                split_bf16x2(v, hi[j], lo[j]);
            }
            // high parts of tokens s0.. at columns s0.., of s0 + 16.. at s0 + 8..; low parts 16 further
            tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)s0, hi);
            tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)(s0 + 16), lo);
        }
        tmem_st_wait();
    };
    // O of the chunk: from tensor memory (row 16 q + (lane & 15), columns 32 hf + 16 (lane >> 4)
    // + 0..15) into a [64][64] fp32 staging tile over the stage's Q~ / K~ high parts (dead once
    // the products have run; 16-byte chunks XOR-ed with the row), then whole rows to global
    // memory (a warp stores one row per instruction)
    auto write_out = [&](int stage, int chunk) {
        const long long r0 = row0_of(chunk);
        float *ot = reinterpret_cast<float *>(smem + stage * C::STAGE + C::OFF_Q);
        {
            const int r = 16 * q + (lane & 15), c0 = 32 * hf + 16 * (lane >> 4);
            uint32_t o[16];
            tmem_ld16x2(tmem + tlane + C::C_O + (uint32_t)(32 * hf), o);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int ch = ((c0 >> 2) + c4) ^ (r & 15);
                *reinterpret_cast<float4 *>(ot + r * 64 + ch * 4) =
                    make_float4(__uint_as_float(o[4 * c4]), __uint_as_float(o[4 * c4 + 1]),
                                __uint_as_float(o[4 * c4 + 2]), __uint_as_float(o[4 * c4 + 3]));
            }
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < kGlaTc * 32 / kGlaTcThreads; ++it) {
            const int idx = tid + it * kGlaTcThreads;
            const int r = idx >> 5, c2 = idx & 31;
            const long long t = r0 + r;  // array row
            if (t >= 0 && t < p.T) {
                const int ch = (c2 >> 1) ^ (r & 15);
                const float2 v = *reinterpret_cast<const float2 *>(ot + r * 64 + ch * 4 + (c2 & 1) * 2);
                *reinterpret_cast<float2 *>(p.o + ((size_t)bh * p.T + t) * p.DV + zb * 64 + 2 * c2) = v;
            }
        }
    };
    // operands written by the threads (and cp.async data) -> the tensor core: every thread fences
    // its writes, the block synchronises, and warp 0 issues
    auto hand_to_tc = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    // ------------------------------------------------ phase 1: the segment's affine pair
#pragma unroll
    for (int j = 0; j < SC; ++j) S[j] = 0.f;
    float la_seg = 0.f;  // thread cdim >= 0: log2 of alpha_seg[cdim]
    // A chunk's in-chunk sums are formed while the tensor cores run the chunk before it.
    load_stage(0, c_begin, false);
    if (nc > 1) load_stage(1, c_begin + 1, false);
    stage_ready(0);
    la_seg += cumulate(0, c_begin);
    __syncthreads();
    for (int i = 0; i < nc; ++i) {
        const int stage = i & 1;
        scale_operands(stage, false);
        state_to_mid(stage);
        hand_to_tc();
        if (warp == 0) {
            issue_u(stage);
            mma_commit_w(barA);
        }
        if (i + 1 < nc) {
            stage_ready(stage ^ 1);
            la_seg += cumulate(stage ^ 1, c_begin + i + 1);
        }
        waitA();
        tc_fence_after();
        state_finish(stage);
        fence_async_smem();  // this thread's writes to the stage before its reload
        tc_fence_before();
        __syncthreads();  // the stage and the state product are consumed
        if (i + 2 < nc) load_stage(stage, c_begin + i + 2, false);
    }

    // ------------------------------------------------ look-back for the incoming state
    constexpr int TILES = SC / 4;
    auto ws_index = [&](size_t u, int tile) {
        return u * (size_t)(TILES * kGlaTcThreads) + (size_t)tile * kGlaTcThreads + tid;
    };
    float Sin[SC];
#pragma unroll
    for (int j = 0; j < SC; ++j) Sin[j] = 0.f;
    auto add_state0 = [&](float scale) {
        if (p.S0 == nullptr) return;
#pragma unroll
        for (int j = 0; j < SC; ++j)
            Sin[j] = fmaf(scale, __ldg(p.S0 + ((size_t)bh * DK + srow) * p.DV + zb * 64 + scol(j)), Sin[j]);
    };
    if (cdim >= 0) alpha_s[cdim] = ex2(la_seg);
    if (seg == 0) {
        add_state0(1.f);
    } else {
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl)
            __stcg(p.agg + ws_index(unit, tl), make_float4(S[4 * tl], S[4 * tl + 1], S[4 * tl + 2], S[4 * tl + 3]));
        if (cdim >= 0) __stcg(p.alpha + unit * DK + cdim, ex2(la_seg));
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(p.flags + unit, 1u);
        float accA = 1.f;  // the decay of this thread's row since the segment's start
        int j = seg - 1;
        while (true) {
            const size_t up = ((size_t)j * p.BH + bh) * p.nzb + zb;
            if (tid == 0) s_flag = wait_flag(p.flags + up, p.hdr, 62u);
            __syncthreads();
            const unsigned int f = s_flag;
            __syncthreads();
            if (f != 1u && f != 2u) break;  // the wait gave up (recorded in the header)
            const float4 *src = (f == 2u) ? p.incl : p.agg;
#pragma unroll
            for (int tl = 0; tl < TILES; ++tl) {
                const float4 v = ld_cg4(src + ws_index(up, tl));
                Sin[4 * tl] = fmaf(accA, v.x, Sin[4 * tl]);
                Sin[4 * tl + 1] = fmaf(accA, v.y, Sin[4 * tl + 1]);
                Sin[4 * tl + 2] = fmaf(accA, v.z, Sin[4 * tl + 2]);
                Sin[4 * tl + 3] = fmaf(accA, v.w, Sin[4 * tl + 3]);
            }
            if (f == 2u) break;
            accA *= ld_cg(p.alpha + up * DK + srow);
            if (--j < 0) {
                add_state0(accA);
                break;
            }
        }
    }
    __syncthreads();  // alpha_s visible
    if (seg != p.n_seg - 1) {
        // inclusive state at the segment's end: diag(alpha_seg) S_in + dS_seg
        const float a = alpha_s[srow];
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl)
            __stcg(p.incl + ws_index(unit, tl),
                   make_float4(fmaf(a, Sin[4 * tl], S[4 * tl]), fmaf(a, Sin[4 * tl + 1], S[4 * tl + 1]),
                               fmaf(a, Sin[4 * tl + 2], S[4 * tl + 2]), fmaf(a, Sin[4 * tl + 3], S[4 * tl + 3])));
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(p.flags + unit, 2u);
    }
    if (p.seg_out != nullptr) {  // this segment's incoming state, for a later traversal
        float4 *dst = reinterpret_cast<float4 *>(p.seg_out + (((size_t)seg * p.BH + bh) * DK + srow) * p.DV +
                                                 zb * 64 + scol(0));
#pragma unroll
        for (int tl = 0; tl < TILES; ++tl)
            __stcg(dst + tl, make_float4(Sin[4 * tl], Sin[4 * tl + 1], Sin[4 * tl + 2], Sin[4 * tl + 3]));
    }

    // ------------------------------------------------ phase 2: outputs from the true state
#pragma unroll
    for (int j = 0; j < SC; ++j) S[j] = Sin[j];
    load_stage(0, c_begin, true);
    if (nc > 1) load_stage(1, c_begin + 1, true);
    stage_ready(0);
    cumulate(0, c_begin);
    __syncthreads();
    for (int i = 0; i < nc; ++i) {
        const int stage = i & 1;
        scale_operands(stage, true);
        state_to_mid(stage);
        write_sb();
        hand_to_tc();
        if (warp == 0) {
            issue_p_o(stage);
            issue_u(stage);
            mma_commit_w(barA);
        }
        if (i + 1 < nc) {
            stage_ready(stage ^ 1);
            cumulate(stage ^ 1, c_begin + i + 1);
        }
        waitA();
        tc_fence_after();
        mask_scores();
        tc_fence_before();
        __syncthreads();  // the masked parts are in tensor memory
        tc_fence_after();
        if (warp == 0) {
            issue_pv(stage);
            mma_commit_w(barB);
        }
        state_finish(stage);
        waitB();
        tc_fence_after();
        write_out(stage, c_begin + i);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();  // the stage and the accumulators are consumed
        if (i + 2 < nc) load_stage(stage, c_begin + i + 2, true);
    }

    if (seg == p.n_seg - 1 && p.ST != nullptr) {
        // reversed: the state before token 0 of the arrays, decayed by a_0
        const float f = REV ? __expf(__ldg(Gb + srow)) : 1.f;
#pragma unroll
        for (int j = 0; j < SC; ++j) p.ST[((size_t)bh * DK + srow) * p.DV + zb * 64 + scol(j)] = f * S[j];
    }
    if (timed_out) {
        atomicOr(&p.hdr->error, kErrTimeout);
        atomicExch(&p.hdr->where, 63u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// ----------------------------------------------------------------- backward: decay on the output columns
// The gradients of the queries and keys carry the decay of the output's own
// column (key dimension i) rather than inside a contraction:
//   dq_r[i] = sum_{s<=r} (do_r . v_s) k_s[i] 2^(c_r[i] - c_s[i]) + 2^(c_r[i]) (do_r S_prev^T)[i]
// With Z~ = Z (.) 2^(c_m - c) and S' = diag(2^c_m) S this is
//   OUT = 2^(c - c_m) (.) [ ((X Y^T) . M) Z~ + X S'^T ]
//   S  <- diag(2^(c_L - c_m)) (S' + Z~^T Y)
// in the roles  dQ: X = dO, Y = V, Z = K, S = the forward state from S0;
//               dK (reversed traversal): X = V, Y = dO, Z = Q, S = the adjoint state from dST.
// X Y^T takes exact bf16 inputs (one product); the masked scores and Z~ are
// split into two bf16 parts (three products), S' too (two products with X).
// A block owns 64 output columns (key dimensions zb*64..) and the state rows
// of those dimensions, [64][DV].
struct GlaBArgs {
    const bf16 *x, *y, *z;  // x, y: [BH][T][DV]; z: [BH][T][DK]
    const float *g;         // [BH][T][DK] natural-log decays
    const float *S0;        // [BH][DK][DV] or NULL
    float *out;             // [BH][T][DK]
    const float *fs_dot;    // [BH][DK][DV] or NULL: each final state row dotted with its row here
    float *fs_part;         // [BH][DK]
    int rev;
    int BH, DK, nzb, n_chunks, seg_chunks, n_seg;
    long long T;
    WsHeader *hdr;
    unsigned int *flags;
    float *alpha;  // [unit][64]
    float4 *agg, *incl;
    // [n_seg][BH][DK][DV] or NULL: the state entering each segment (in traversal order), saved
    // by an earlier traversal with the same segments; phase 1 and the look-back are then skipped
    const float *seg_in;
};

// ----------------------------------------------------------------- dQ / dK traversal on tcgen05
// The traversal of the equations above on the tensor cores, per 64-token chunk, with Z~ = Z (.) 2^(c_m - c) and S' = diag(2^c_m) S (the
// block's 64 key dimensions; both split into two bf16 parts by the threads):
//     D    = X Y^T                     (M = 64, N = 64, K = DV)   one product (exact inputs)
//     O    = X S'^T                    (M = 64, N = 64, K = DV)   two products
//     U    = Z~^T Y                    (M = 64, N = DV, K = 64)   two products
//     O   += (D . M) Z~                (A from tensor memory)     three products
//     OUT  = 2^(c - c_m) (.) O,  S_next = diag(2^(c_L - c_m)) (S' + U)
// Tiles use the 128-byte swizzle: X, Y K-major ([64 tokens][DV]; Y also the
// MN-major B of U), Z~ MN-major (B of the last product, A of U), S' K-major
// ([64 key dimensions][DV]).  8 warps as in gla_tc_kernel: warps w and w + 4
// read lane quarter w & 3 of tensor memory and split its columns.
template <int DV>
struct GlaQkCfg {
    static constexpr int KB = DV / 64;             // 64-element blocks along the value dimension
    static constexpr int XT_BYTES = KB * 64 * 128;  // a [64 tokens][DV] bf16 operand tile
    static constexpr int Z_BYTES = 64 * 128;        // a [64 tokens][64 key dimensions] bf16 tile
    static constexpr int G_BYTES = 64 * 64 * 4;     // log decays of the 64 key dimensions
    static constexpr int OFF_X = 0;
    static constexpr int OFF_Y = XT_BYTES;
    static constexpr int OFF_Z = 2 * XT_BYTES;
    static constexpr int OFF_G = 2 * XT_BYTES + Z_BYTES;
    static constexpr int STAGE = 2 * XT_BYTES + Z_BYTES + G_BYTES;
    static constexpr int OFF_ZL = 2 * STAGE;             // low part of Z~
    static constexpr int OFF_SH = OFF_ZL + Z_BYTES;      // S' high part, [64 key dimensions][DV] K-major
    static constexpr int OFF_SL = OFF_SH + XT_BYTES;
    static constexpr int OFF_AS = OFF_SL + XT_BYTES;     // alpha of the segment per key dimension [64]
    static constexpr int OFF_FS = OFF_AS + 64 * 4;       // the final-state dot, per column half [2][64]
    static constexpr int OFF_BAR = OFF_FS + 2 * 64 * 4;  // four mbarriers: two products, two stage loads
    static constexpr int SMEM = OFF_BAR + 32 + 1024;     // + alignment slack of the 1024-byte base
    // tensor memory: D, masked D parts, O, U (DV columns)
    static constexpr uint32_t C_D = 0, C_DB = 64, C_O = 128, C_U = 192, TMEM_COLS = 512;
    static constexpr int SC = DV / 4;  // state columns per thread
    static_assert(STAGE % 1024 == 0 && XT_BYTES % 1024 == 0, "1024-byte aligned operand tiles");
    static_assert(2 * XT_BYTES >= 64 * 64 * 4, "the output tile fits over a stage's X and Y");
    static_assert(C_U + DV <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Tensor maps of the traversal operands: X and Y ([BH][T][DV] bf16) and Z ([BH][T][d_k]
// bf16, a 64-column box) in 128-byte-swizzled boxes of 64 tokens x 64 columns, the log decays
// ([BH][T][d_k] fp32) in plain boxes of 64 tokens x 64 dimensions.
struct GlaQkMaps {
    CUtensorMap x, y, z, g;
};

// Stages filled by TMA as in gla_tc_kernel; REV (the dK traversal): row j of a stage holds
// traversal position 63 - j.
template <int DV, bool REV>
__global__ void __launch_bounds__(kGlaTcThreads, 1)
    gla_tc_qk_kernel(const GlaBArgs p, const __grid_constant__ GlaQkMaps maps) {
    using C = GlaQkCfg<DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    __shared__ uint32_t s_tmem;
    __shared__ unsigned int s_ticket, s_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t barA = sbase + C::OFF_BAR, barB = barA + 8, barL = barA + 16;  // barL + 8 stage

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 0) {
        mbar_init(barA, 1);
        mbar_init(barB, 1);
        mbar_init(barL, 1);
        mbar_init(barL + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ticket = atomicAdd(&p.hdr->ticket[0], 1u);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int q = warp & 3, hf = warp >> 2;
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    const unsigned int tk = s_ticket;
    const int per_seg = p.BH * p.nzb;
    const int seg = (int)(tk / per_seg);
    const int bh = (int)(tk % per_seg) / p.nzb;
    const int zb = (int)(tk % per_seg) % p.nzb;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
    const int nc = c_end - c_begin;
    const size_t unit = ((size_t)seg * p.BH + bh) * p.nzb + zb;
    bool timed_out = false;
    uint32_t phA = 0u, phB = 0u;
    auto waitA = [&]() {
        if (!mbar_wait(barA, phA)) timed_out = true;
        phA ^= 1u;
    };
    auto waitB = [&]() {
        if (!mbar_wait(barB, phB)) timed_out = true;
        phB ^= 1u;
    };
    uint32_t phL = 0u;  // bit s: parity of stage s's next load
    auto stage_ready = [&](int stage) {
        if (!mbar_wait(barL + 8u * (uint32_t)stage, (phL >> stage) & 1u)) timed_out = true;
        phL ^= 1u << stage;
    };
    // stage rows of the chunk's midpoint token and of its last token
    constexpr int MID = REV ? kGlaTc - 1 - kGlaMid : kGlaMid;
    constexpr int LAST = REV ? 0 : kGlaTc - 1;
    float *alpha_s = reinterpret_cast<float *>(smem + C::OFF_AS);

    // array row of a chunk's stage row 0 (reversed: of its last traversal position)
    auto row0_of = [&](int chunk) {
        return REV ? p.T - (long long)kGlaTc * (chunk + 1) : (long long)kGlaTc * chunk;
    };
    // the reversed traversal's decay of position t' is array token T - t': its G tile starts a row later
    auto load_stage = [&](int stage, int chunk, bool withX) {
        if (tid != 0) return;
        const uint32_t bar = barL + 8u * (uint32_t)stage, s0 = smem_u32(smem + stage * C::STAGE);
        mbar_expect_tx(bar, (uint32_t)((withX ? 2 : 1) * C::XT_BYTES + C::Z_BYTES + C::G_BYTES));
        const int y = (int)row0_of(chunk);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(s0 + C::OFF_Y + kb * 8192, &maps.y, kb * 64, y, bh, bar);
            if (withX) tma_load_3d(s0 + C::OFF_X + kb * 8192, &maps.x, kb * 64, y, bh, bar);
        }
        tma_load_3d(s0 + C::OFF_Z, &maps.z, zb * 64, y, bh, bar);
        tma_load_3d(s0 + C::OFF_G, &maps.g, zb * 64, REV ? y + 1 : y, bh, bar);
    };
    // in-chunk cumulative log2 decays in traversal order (positions past the end decay by
    // nothing), by the last 64 threads (they issue no products): thread cdim >= 0 scans cdim
    const int cdim = tid - (kGlaTcThreads - 64);
    auto cumulate = [&](int stage, int chunk) {
        float *G = reinterpret_cast<float *>(smem + stage * C::STAGE + C::OFF_G);
        float total = 0.f;
        if (cdim >= 0) {
            const long long n_tok = p.T - (long long)kGlaTc * chunk;
            float run = 0.f, lo = 0.f, hi = 0.f;
            bool finite = true;
#pragma unroll 8
            for (int t = 0; t < kGlaTc; ++t) {
                const int row = REV ? kGlaTc - 1 - t : t;
                const float l = (REV && t >= n_tok) ? 0.f : G[row * 64 + cdim];
                finite = finite && isfinite(l);
                run += l * kGlaLog2e;
                G[row * 64 + cdim] = run;
                lo = fminf(lo, run);
                hi = fmaxf(hi, run);
            }
            const float cm = G[MID * 64 + cdim];
            if (!finite || hi - cm > kGlaSpan || cm - lo > kGlaSpan || cm > kGlaSpan)
                atomicOr(&p.hdr->error, kErrRange);
            total = run;
        }
        return total;
    };
    // Z~ = Z 2^(c_m - c): high part over Z, low part in ZL
    auto scale_z = [&](int stage) {
        uint8_t *st = smem + stage * C::STAGE;
        const float *G = reinterpret_cast<const float *>(st + C::OFF_G);
        // a thread keeps its 8 key dimensions (the same in every round) and steps over rows
        const int c16 = tid & 7;
        float2 cm[4];  // c_m of the thread's dimensions
        {
            const float4 *cmid = reinterpret_cast<const float4 *>(G + MID * 64 + c16 * 8);
            const float4 ma = cmid[0], mb = cmid[1];
            cm[0] = make_float2(ma.x, ma.y);
            cm[1] = make_float2(ma.z, ma.w);
            cm[2] = make_float2(mb.x, mb.y);
            cm[3] = make_float2(mb.z, mb.w);
        }
#pragma unroll
        for (int it = 0; it < kGlaTc * 8 / kGlaTcThreads; ++it) {
            const int row = (tid >> 3) + it * (kGlaTcThreads / 8);
            const float4 *crow = reinterpret_cast<const float4 *>(G + row * 64 + c16 * 8);
            const float4 a = crow[0], b = crow[1];
            const float2 nc[4] = {make_float2(-a.x, -a.y), make_float2(-a.z, -a.w), make_float2(-b.x, -b.y),
                                  make_float2(-b.z, -b.w)};
            const uint32_t off = sw128(row, c16 * 8);
            const uint4 zv = *reinterpret_cast<const uint4 *>(st + C::OFF_Z + off);
            const uint32_t w[4] = {zv.x, zv.y, zv.z, zv.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 d = __fadd2_rn(cm[e], nc[e]);  // c_m - c
                split_bf16x2(__fmul2_rn(unpack_bf16(w[e]), make_float2(ex2(d.x), ex2(d.y))), hi[e], lo[e]);
            }
            *reinterpret_cast<uint4 *>(st + C::OFF_Z + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(smem + C::OFF_ZL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };


    // This thread's state: key dimension srow (row of the 64-row accumulator U) and SC columns of
    // the value half hf, in runs of 16: 64-row layout, paired-half shape.
    constexpr int SC = C::SC;
    const int srow = 16 * q + (lane & 15);
    auto scol = [&](int j) { return (DV / 2) * hf + ((j >> 4) << 5) + 16 * (lane >> 4) + (j & 15); };
    float S[SC];
    auto load_u = [&](float (&u)[SC]) {
#pragma unroll
        for (int g32 = 0; g32 < SC / 16; ++g32) {
            uint32_t r[16];
            tmem_ld16x2(tmem + tlane + C::C_U + (uint32_t)((DV / 2) * hf + 32 * g32), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) u[16 * g32 + j] = __uint_as_float(r[j]);
        }
    };
    auto state_to_mid = [&](int stage) {
        const float *G = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_G);
        const float f = ex2(G[MID * 64 + srow]);
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] *= f;
    };
    // S' as two bf16 parts, K-major [64 key dimensions][DV] (the B operand of X S'^T)
    auto write_sb = [&]() {
#pragma unroll
        for (int j8 = 0; j8 < SC / 8; ++j8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(make_float2(S[8 * j8 + 2 * e], S[8 * j8 + 2 * e + 1]), hi[e], lo[e]);
            const int col = scol(8 * j8);
            const uint32_t off = (uint32_t)((col >> 6) * 8192) + sw128(srow, col & 63);
            *reinterpret_cast<uint4 *>(smem + C::OFF_SH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(smem + C::OFF_SL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };
    auto state_finish = [&](int stage) {
        const float *G = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_G);
        const float f = ex2(G[LAST * 64 + srow] - G[MID * 64 + srow]);
        float u[SC];
        load_u(u);
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] = f * (S[j] + u[j]);
    };

    // ---- descriptors
    auto kdesc = [&](uint32_t off) { return smem_desc(sbase + off, 16, 1024); };     // K-major
    auto mndesc = [&](uint32_t off) { return smem_desc(sbase + off, 8192, 1024); };  // MN-major
    auto kstep_k = [&](int kk) { return (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4); };
    auto kstep_mn = [&](int kk) { return (uint64_t)((kk * 2048) >> 4); };
    constexpr uint32_t id_d = idesc_bf16(64, 64, 0, 0);   // D = X Y^T
    constexpr uint32_t id_o = idesc_bf16(64, 64, 0, 0);   // O = X S'^T (S' K-major)
    constexpr uint32_t id_u = idesc_bf16(64, DV, 1, 1);   // U = Z~^T Y
    constexpr uint32_t id_i = idesc_bf16(64, 64, 0, 1);   // O += (D . M) Z~
    auto issue_u = [&](int stage) {
        const uint32_t so = (uint32_t)(stage * C::STAGE);
        const uint64_t b0 = mndesc(so + C::OFF_Y);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const uint64_t a0 = mndesc(part ? C::OFF_ZL : so + C::OFF_Z);
#pragma unroll
            for (int kk = 0; kk < kGlaTc / 16; ++kk)
                mma_ss_w(tmem + C::C_U, a0 + kstep_mn(kk), b0 + kstep_mn(kk), id_u, (part | kk) ? 1u : 0u);
        }
    };
    auto issue_d_o = [&](int stage) {
        const uint32_t so = (uint32_t)(stage * C::STAGE);
        const uint64_t a0 = kdesc(so + C::OFF_X), by = kdesc(so + C::OFF_Y);
        const uint64_t sh = kdesc(C::OFF_SH), sl = kdesc(C::OFF_SL);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
            mma_ss_w(tmem + C::C_D, a0 + kstep_k(kk), by + kstep_k(kk), id_d, kk ? 1u : 0u);
            mma_ss_w(tmem + C::C_O, a0 + kstep_k(kk), sh + kstep_k(kk), id_o, kk ? 1u : 0u);
            mma_ss_w(tmem + C::C_O, a0 + kstep_k(kk), sl + kstep_k(kk), id_o, 1u);
        }
    };
    // O += (D . M)_hi Z~_hi + (D . M)_hi Z~_lo + (D . M)_lo Z~_hi
    auto issue_intra = [&](int stage) {
        const uint64_t zh = mndesc((uint32_t)(stage * C::STAGE) + C::OFF_Z), zl = mndesc(C::OFF_ZL);
#pragma unroll
        for (int part = 0; part < 3; ++part) {
            const int apart = (part == 2) ? 1 : 0;
            const uint64_t b0 = (part == 1) ? zl : zh;
#pragma unroll
            for (int kk = 0; kk < kGlaTc / 16; ++kk) {
                const uint32_t acol = C::C_DB + (uint32_t)(kk >> 1) * 32 + apart * 16 + (kk & 1) * 8;
                mma_ts_w(tmem + C::C_O, tmem + acol, b0 + kstep_mn(kk), id_i, 1u);
            }
        }
    };
    auto mask_d = [&]() {
        const int r = 16 * q + (lane & 15);
        const int s0 = hf * 32;
        uint32_t pr[16];
        tmem_ld16x2(tmem + tlane + C::C_D + (uint32_t)s0, pr);
        tmem_ld_wait();
        const int sb = s0 + 16 * (lane >> 4);
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = sb + 2 * j;
            float2 v = make_float2(__uint_as_float(pr[2 * j]), __uint_as_float(pr[2 * j + 1]));
            if (REV ? s < r : s > r) v.x = 0.f;  // reversed stage rows: keep s >= r
            if (REV ? s + 1 < r : s + 1 > r) v.y = 0.f;
            split_bf16x2(v, hi[j], lo[j]);
        }
        tmem_st8x2(tmem + tlane + C::C_DB + (uint32_t)s0, hi);
        tmem_st8x2(tmem + tlane + C::C_DB + (uint32_t)(s0 + 16), lo);
        tmem_st_wait();
    };
    // OUT = 2^(c_r - c_m) O per (token r, key dimension): O staged over the stage's X and Y (dead
    // once the products have run; 16-byte chunks XOR-ed with the row), then scaled and written a
    // row per warp (the row's decays read as one contiguous run per warp: no bank conflicts)
    auto write_out = [&](int stage, int chunk) {
        const long long r0 = row0_of(chunk);
        const float *G = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_G);
        float *ot = reinterpret_cast<float *>(smem + stage * C::STAGE + C::OFF_X);
        {
            const int r = 16 * q + (lane & 15), c0 = 32 * hf + 16 * (lane >> 4);
            uint32_t o[16];
            tmem_ld16x2(tmem + tlane + C::C_O + (uint32_t)(32 * hf), o);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int ch = ((c0 >> 2) + c4) ^ (r & 15);
                *reinterpret_cast<uint4 *>(ot + r * 64 + ch * 4) =
                    make_uint4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
            }
        }
        __syncthreads();
        const float2 cm = *reinterpret_cast<const float2 *>(G + MID * 64 + 2 * lane);  // the same columns every round
#pragma unroll
        for (int it = 0; it < kGlaTc * 32 / kGlaTcThreads; ++it) {
            const int idx = tid + it * kGlaTcThreads;
            const int r = idx >> 5, c2 = idx & 31;
            const long long t = r0 + r;  // array row
            if (t >= 0 && t < p.T) {
                const int ch = (c2 >> 1) ^ (r & 15);
                const float2 v = *reinterpret_cast<const float2 *>(ot + r * 64 + ch * 4 + (c2 & 1) * 2);
                const float2 cr = *reinterpret_cast<const float2 *>(G + r * 64 + 2 * c2);
                *reinterpret_cast<float2 *>(p.out + ((size_t)bh * p.T + t) * p.DK + zb * 64 + 2 * c2) =
                    make_float2(v.x * ex2(cr.x - cm.x), v.y * ex2(cr.y - cm.y));
            }
        }
    };

    auto hand_to_tc = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    constexpr int TILES = SC / 4;
    float Sin[SC];
    if (p.seg_in != nullptr) {
        // the incoming state saved by an earlier traversal: no phase 1, no look-back
        const float *src = p.seg_in + (((size_t)seg * p.BH + bh) * p.DK + zb * 64 + srow) * DV;
#pragma unroll
        for (int j = 0; j < SC; ++j) Sin[j] = __ldg(src + scol(j));
    } else {
        // ------------------------------------------------ phase 1
#pragma unroll
        for (int j = 0; j < SC; ++j) S[j] = 0.f;
        float la_seg = 0.f;
        // a chunk's in-chunk sums are formed while the tensor cores run the chunk before it
        load_stage(0, c_begin, false);
        if (nc > 1) load_stage(1, c_begin + 1, false);
        stage_ready(0);
        la_seg += cumulate(0, c_begin);
        __syncthreads();
        for (int i = 0; i < nc; ++i) {
            const int stage = i & 1;
            scale_z(stage);
            state_to_mid(stage);
            hand_to_tc();
            if (warp == 0) {
                issue_u(stage);
                mma_commit_w(barA);
            }
            if (i + 1 < nc) {
                stage_ready(stage ^ 1);
                la_seg += cumulate(stage ^ 1, c_begin + i + 1);
            }
            waitA();
            tc_fence_after();
            state_finish(stage);
            fence_async_smem();  // this thread's writes to the stage before its reload
            tc_fence_before();
            __syncthreads();
            if (i + 2 < nc) load_stage(stage, c_begin + i + 2, false);
        }

        // ------------------------------------------------ look-back
        auto ws_index = [&](size_t u, int tile) {
            return u * (size_t)(TILES * kGlaTcThreads) + (size_t)tile * kGlaTcThreads + tid;
        };
#pragma unroll
        for (int j = 0; j < SC; ++j) Sin[j] = 0.f;
        auto add_state0 = [&](float scale) {
            if (p.S0 == nullptr) return;
#pragma unroll
            for (int j = 0; j < SC; ++j)
                Sin[j] = fmaf(scale, __ldg(p.S0 + ((size_t)bh * p.DK + zb * 64 + srow) * DV + scol(j)), Sin[j]);
        };
        if (cdim >= 0) alpha_s[cdim] = ex2(la_seg);
        if (seg == 0) {
            add_state0(1.f);
        } else {
#pragma unroll
            for (int tl = 0; tl < TILES; ++tl)
                __stcg(p.agg + ws_index(unit, tl), make_float4(S[4 * tl], S[4 * tl + 1], S[4 * tl + 2], S[4 * tl + 3]));
            if (cdim >= 0) __stcg(p.alpha + unit * 64 + cdim, ex2(la_seg));
            __threadfence();
            __syncthreads();
            if (tid == 0) st_release(p.flags + unit, 1u);
            float accA = 1.f;
            int j = seg - 1;
            while (true) {
                const size_t up = ((size_t)j * p.BH + bh) * p.nzb + zb;
                if (tid == 0) s_flag = wait_flag(p.flags + up, p.hdr, 64u);
                __syncthreads();
                const unsigned int f = s_flag;
                __syncthreads();
                if (f != 1u && f != 2u) break;
                const float4 *src = (f == 2u) ? p.incl : p.agg;
#pragma unroll
                for (int tl = 0; tl < TILES; ++tl) {
                    const float4 v = ld_cg4(src + ws_index(up, tl));
                    Sin[4 * tl] = fmaf(accA, v.x, Sin[4 * tl]);
                    Sin[4 * tl + 1] = fmaf(accA, v.y, Sin[4 * tl + 1]);
                    Sin[4 * tl + 2] = fmaf(accA, v.z, Sin[4 * tl + 2]);
                    Sin[4 * tl + 3] = fmaf(accA, v.w, Sin[4 * tl + 3]);
                }
                if (f == 2u) break;
                accA *= ld_cg(p.alpha + up * 64 + srow);
                if (--j < 0) {
                    add_state0(accA);
                    break;
                }
            }
        }
        __syncthreads();
        if (seg != p.n_seg - 1) {
            const float a = alpha_s[srow];
#pragma unroll
            for (int tl = 0; tl < TILES; ++tl)
                __stcg(p.incl + ws_index(unit, tl),
                       make_float4(fmaf(a, Sin[4 * tl], S[4 * tl]), fmaf(a, Sin[4 * tl + 1], S[4 * tl + 1]),
                                   fmaf(a, Sin[4 * tl + 2], S[4 * tl + 2]), fmaf(a, Sin[4 * tl + 3], S[4 * tl + 3])));
            __threadfence();
            __syncthreads();
            if (tid == 0) st_release(p.flags + unit, 2u);
        }
    }  // phase 1 and look-back

    // ------------------------------------------------ phase 2
#pragma unroll
    for (int j = 0; j < SC; ++j) S[j] = Sin[j];
    load_stage(0, c_begin, true);
    if (nc > 1) load_stage(1, c_begin + 1, true);
    stage_ready(0);
    cumulate(0, c_begin);
    __syncthreads();
    for (int i = 0; i < nc; ++i) {
        const int stage = i & 1;
        scale_z(stage);
        state_to_mid(stage);
        write_sb();
        hand_to_tc();
        if (warp == 0) {
            issue_d_o(stage);
            issue_u(stage);
            mma_commit_w(barA);
        }
        if (i + 1 < nc) {
            stage_ready(stage ^ 1);
            cumulate(stage ^ 1, c_begin + i + 1);
        }
        waitA();
        tc_fence_after();
        mask_d();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0) {
            issue_intra(stage);
            mma_commit_w(barB);
        }
        state_finish(stage);
        waitB();
        tc_fence_after();
        write_out(stage, c_begin + i);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (i + 2 < nc) load_stage(stage, c_begin + i + 2, true);
    }

    // the final state's rows dotted with fs_dot (the decay gradient's final-state term): the
    // paired halves of a warp, then the two column halves, summed through shared memory
    if (seg == p.n_seg - 1 && p.fs_part != nullptr) {
        float *fsx = reinterpret_cast<float *>(smem + C::OFF_FS);
        float acc = 0.f;
        if (p.fs_dot != nullptr) {
#pragma unroll
            for (int j = 0; j < SC; ++j)
                acc = fmaf(S[j], __ldg(p.fs_dot + ((size_t)bh * p.DK + zb * 64 + srow) * DV + scol(j)), acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        if (lane < 16) fsx[hf * 64 + srow] = acc;
        __syncthreads();
        if (tid < 64) p.fs_part[(size_t)bh * p.DK + zb * 64 + tid] = fsx[tid] + fsx[64 + tid];
    }
    if (timed_out) {
        atomicOr(&p.hdr->error, kErrTimeout);
        atomicExch(&p.hdr->where, 65u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// ----------------------------------------------------------------- backward: decay gradient
// Closed form per key dimension ("The backward pass of linear attention",
// Yang et al.'s form for gated linear attention):
//   dlog a_u[i] = sum_{t>=u} (q_t[i] dq_t[i] - k_t[i] dk_t[i]) + fs[i],
// fs[i] = sum_j dST[i][j] S_T[i][j].  A reverse scan over tiles of
// kGlaDlTile tokens: per-tile column sums first, then (one short pass per
// batch and head) the sum of every later tile and fs for each tile, then
// each tile's suffix sums from it.  Thread = key dimension (coalesced rows);
// fixed summation order; loops unrolled so a thread's loads are in flight
// together.
constexpr int kGlaDlTile = 128;

__global__ void gla_dlog_tile_sums_kernel(const bf16 *__restrict__ q, const float *__restrict__ dq,
                                          const bf16 *__restrict__ k, const float *__restrict__ dk,
                                          float *__restrict__ tsum, int DK, long long T, int n_tiles) {
    const int tile = (int)(blockIdx.x % (unsigned)n_tiles);
    const size_t bh = blockIdx.x / (unsigned)n_tiles;
    const int i = threadIdx.x;
    const long long t0 = (long long)tile * kGlaDlTile;
    const long long t1 = min(t0 + kGlaDlTile, T);
    float acc = 0.f;
#pragma unroll 8
    for (long long t = t0; t < t1; ++t) {
        const size_t x = (bh * T + t) * DK + i;
        acc += __bfloat162float(__ldg(q + x)) * __ldg(dq + x) - __bfloat162float(__ldg(k + x)) * __ldg(dk + x);
    }
    tsum[(bh * n_tiles + tile) * DK + i] = acc;
}

// The tile sums of one (batch, head) become, in place and in the same fixed order, the sums of
// every later tile plus the final-state term: what each tile's suffix scan starts from.
__global__ void gla_dlog_tile_suffix_kernel(float *__restrict__ tsum, const float *__restrict__ fs, int DK,
                                            int n_tiles) {
    const size_t bh = blockIdx.x;
    const int i = threadIdx.x;
    float run = fs ? fs[bh * DK + i] : 0.f;
#pragma unroll 4
    for (int j = n_tiles - 1; j >= 0; --j) {
        float *x = tsum + (bh * n_tiles + j) * DK + i;
        const float v = *x;
        *x = run;
        run += v;
    }
}

__global__ void gla_dlog_finalize_kernel(const bf16 *__restrict__ q, const float *__restrict__ dq,
                                         const bf16 *__restrict__ k, const float *__restrict__ dk,
                                         const float *__restrict__ tsum, float *__restrict__ dlog, int DK,
                                         long long T, int n_tiles) {
    const int tile = (int)(blockIdx.x % (unsigned)n_tiles);
    const size_t bh = blockIdx.x / (unsigned)n_tiles;
    const int i = threadIdx.x;
    float run = tsum[(bh * n_tiles + tile) * DK + i];  // the later tiles and the final-state term
    const long long t0 = (long long)tile * kGlaDlTile;
#pragma unroll 8
    for (long long t = min(t0 + kGlaDlTile, T) - 1; t >= t0; --t) {
        const size_t x = (bh * T + t) * DK + i;
        run += __bfloat162float(__ldg(q + x)) * __ldg(dq + x) - __bfloat162float(__ldg(k + x)) * __ldg(dk + x);
        dlog[x] = run;
    }
}

// The same two passes with 8 key dimensions per thread (16-byte loads of q and k, 32-byte ones of
// dq and dk: eight times a scalar thread's bytes in flight), DK / 8 threads per (batch-head,
// tile) unit and 128 / (DK / 8) units per block; the sums per dimension in the same token order.
// Taken when dq, dk and dlog are 16-byte aligned.
constexpr int kGlaDl8Threads = 128;

__device__ __forceinline__ void gla_dl8_term(const bf16 *q, const float *dq, const bf16 *k, const float *dk, size_t x,
                                             float (&u)[8]) {
    const uint4 qv = __ldg(reinterpret_cast<const uint4 *>(q + x));
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k + x));
    const float4 a0 = __ldg(reinterpret_cast<const float4 *>(dq + x)), a1 = __ldg(reinterpret_cast<const float4 *>(dq + x + 4));
    const float4 b0 = __ldg(reinterpret_cast<const float4 *>(dk + x)), b1 = __ldg(reinterpret_cast<const float4 *>(dk + x + 4));
    const float dqv[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float dkv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 qq = unpack_bf16(qw[e]), kk = unpack_bf16(kw[e]);
        u[2 * e] = qq.x * dqv[2 * e] - kk.x * dkv[2 * e];
        u[2 * e + 1] = qq.y * dqv[2 * e + 1] - kk.y * dkv[2 * e + 1];
    }
}

__global__ void __launch_bounds__(kGlaDl8Threads)
gla_dlog_tile_sums8_kernel(const bf16 *__restrict__ q, const float *__restrict__ dq, const bf16 *__restrict__ k,
                           const float *__restrict__ dk, float *__restrict__ tsum, int DK, long long T, int n_tiles,
                           long long n_units) {
    const int tpu = DK / 8;
    const long long unit = (long long)blockIdx.x * (kGlaDl8Threads / tpu) + threadIdx.x / tpu;
    if (unit >= n_units) return;
    const int j = threadIdx.x % tpu;
    const int tile = (int)(unit % n_tiles);
    const size_t bh = (size_t)(unit / n_tiles);
    const long long t0 = (long long)tile * kGlaDlTile;
    const long long t1 = min(t0 + kGlaDlTile, T);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (long long t = t0; t < t1; ++t) {
        float u[8];
        gla_dl8_term(q, dq, k, dk, (bh * T + t) * DK + 8 * j, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += u[e];
    }
    float4 *dst = reinterpret_cast<float4 *>(tsum + (bh * n_tiles + tile) * DK + 8 * j);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__global__ void __launch_bounds__(kGlaDl8Threads)
gla_dlog_finalize8_kernel(const bf16 *__restrict__ q, const float *__restrict__ dq, const bf16 *__restrict__ k,
                          const float *__restrict__ dk, const float *__restrict__ tsum, float *__restrict__ dlog, int DK,
                          long long T, int n_tiles, long long n_units) {
    const int tpu = DK / 8;
    const long long unit = (long long)blockIdx.x * (kGlaDl8Threads / tpu) + threadIdx.x / tpu;
    if (unit >= n_units) return;
    const int j = threadIdx.x % tpu;
    const int tile = (int)(unit % n_tiles);
    const size_t bh = (size_t)(unit / n_tiles);
    float run[8];  // the later tiles and the final-state term
    {
        const float4 *src = reinterpret_cast<const float4 *>(tsum + (bh * n_tiles + tile) * DK + 8 * j);
        const float4 r0 = src[0], r1 = src[1];
        run[0] = r0.x; run[1] = r0.y; run[2] = r0.z; run[3] = r0.w;
        run[4] = r1.x; run[5] = r1.y; run[6] = r1.z; run[7] = r1.w;
    }
    const long long t0 = (long long)tile * kGlaDlTile;
#pragma unroll 8
    for (long long t = min(t0 + kGlaDlTile, T) - 1; t >= t0; --t) {
        const size_t x = (bh * T + t) * DK + 8 * j;
        float u[8];
        gla_dl8_term(q, dq, k, dk, x, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) run[e] += u[e];
        float4 *d = reinterpret_cast<float4 *>(dlog + x);
        d[0] = make_float4(run[0], run[1], run[2], run[3]);
        d[1] = make_float4(run[4], run[5], run[6], run[7]);
    }
}

// ----------------------------------------------------------------- host side
struct GlaPlan {
    int n_chunks, seg_chunks, n_seg, nzb;
    size_t units, off_flags, off_alpha, off_agg, off_incl, total;
};

// Segments of chunks, the same for every traversal of one head's sequence (the forward, dQ, dV,
// dK), so that a state one traversal forms at a segment's start can start another: the largest
// of kGlaSegChoices that still gives kGlaMinBlocks blocks to the traversal with the most column
// blocks (max(d_k, d_v) / 64 per head).
void gla_segments(int64_t BH, int n_chunks, int64_t dk, int64_t dv, int &seg_chunks, int &n_seg) {
    const int64_t nzb = (dk > dv ? dk : dv) / 64;
    seg_chunks = kGlaSegChoices[3];
    for (int c : kGlaSegChoices) {
        if ((long long)((n_chunks + c - 1) / c) * BH * nzb >= kGlaMinBlocks) {
            seg_chunks = c;
            break;
        }
    }
    n_seg = (n_chunks + seg_chunks - 1) / seg_chunks;
    if (n_seg < 1) n_seg = 1;
}

GlaPlan gla_plan(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv) {
    GlaPlan p;
    p.n_chunks = (int)((T + kGlaTc - 1) / kGlaTc);
    p.nzb = (int)(dv / 64);
    const size_t BH = (size_t)B * H;
    gla_segments((int64_t)BH, p.n_chunks, dk, dv, p.seg_chunks, p.n_seg);
    p.units = (size_t)p.n_seg * BH * p.nzb;
    p.off_flags = sizeof(WsHeader);
    p.off_alpha = align_up(p.off_flags + p.units * 4, 256);
    p.off_agg = align_up(p.off_alpha + p.units * (size_t)dk * 4, 256);
    const size_t state_bytes = (size_t)dk * 64 * 4;  // one block's state tiles
    p.off_incl = align_up(p.off_agg + p.units * state_bytes, 256);
    p.total = align_up(p.off_incl + p.units * state_bytes, 256);
    return p;
}

// Sizes the kernel handles: B*H <= 2^24, T < 2^31 (32-bit token coordinates of the tensor-map
// loads), B*H*T <= 2^40, grid below 2^31 blocks.
bool gla_sizes_fit(int64_t B, int64_t H, int64_t T) {
    if (!product_below({B, H}, 16777217.0) || T > kMaxTokens) return false;
    if (!product_below({B, H, T}, 1099511627777.0)) return false;
    const int64_t n_chunks = (T + kGlaTc - 1) / kGlaTc;
    return product_below({B, H, n_chunks, 2}, 2147483648.0);
}

bool gla_supported(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int chunk) {
    return B >= 0 && H >= 0 && T >= 0 && (dk == 64 || dk == 128) && dv > 0 && dv % 64 == 0 && dv <= 1024 &&
           chunk == kGlaTc && gla_sizes_fit(B, H, T);
}


// Backward workspace: the look-back arrays of the largest traversal (reused by the three in
// turn), the final-state term per key dimension and the decay gradient's tile sums.
struct GlaBwdPlan {
    int n_chunks, seg_chunks, n_seg, tiles;
    size_t off_flags, off_alpha, off_agg, off_incl, off_fs, off_tsum, off_seg, total;
};

GlaBwdPlan gla_bwd_plan(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv) {
    GlaBwdPlan p;
    const int64_t BH = B * H;
    p.n_chunks = (int)((T + kGlaTc - 1) / kGlaTc);
    gla_segments(BH, p.n_chunks, dk, dv, p.seg_chunks, p.n_seg);
    const size_t unitsA = (size_t)p.n_seg * BH * (dv / 64), unitsB = (size_t)p.n_seg * BH * (dk / 64);
    const size_t units = unitsA > unitsB ? unitsA : unitsB;
    const size_t alpha_floats = unitsA * dk > unitsB * 64 ? unitsA * dk : unitsB * 64;
    const size_t state_floats = unitsA * dk * 64 > unitsB * 64 * dv ? unitsA * dk * 64 : unitsB * 64 * dv;
    p.tiles = (int)((T + kGlaDlTile - 1) / kGlaDlTile);
    if (p.tiles < 1) p.tiles = 1;
    p.off_flags = sizeof(WsHeader);
    p.off_alpha = align_up(p.off_flags + units * 4, 256);
    p.off_agg = align_up(p.off_alpha + alpha_floats * 4, 256);
    p.off_incl = align_up(p.off_agg + state_floats * 4, 256);
    p.off_fs = align_up(p.off_incl + state_floats * 4, 256);
    p.off_tsum = align_up(p.off_fs + (size_t)BH * dk * 4, 256);
    // the adjoint state entering each segment: saved by the dV traversal, read by the dK one
    p.off_seg = align_up(p.off_tsum + (size_t)BH * p.tiles * dk * 4, 256);
    p.total = p.off_seg + align_up((size_t)p.n_seg * BH * dk * dv * 4, 256);
    return p;
}

bool gla_bwd_supported(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int chunk) {
    return B >= 0 && H >= 0 && T >= 0 && (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && chunk == kGlaTc &&
           gla_sizes_fit(B, H, T) && product_below({B, H, (T + kGlaDlTile - 1) / kGlaDlTile}, 2147483648.0);
}

template <int DV, bool REV>
int launch_gla_bwd_qk_variant(const GlaBArgs &a, const GlaQkMaps &maps, cudaStream_t s, unsigned int grid) {
    using C = GlaQkCfg<DV>;
    static std::atomic<unsigned long long> smem_set{0};  // per template instance
    const int st =
        set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(gla_tc_qk_kernel<DV, REV>), C::SMEM);
    if (st) return st;
    gla_tc_qk_kernel<DV, REV><<<grid, kGlaTcThreads, C::SMEM, s>>>(a, maps);
    return check_launch("gla_tc_qk_kernel");
}

template <int DV>
int launch_gla_bwd_qk(const GlaBArgs &a, cudaStream_t s, unsigned int grid) {
    GlaQkMaps maps;
    memset(&maps, 0, sizeof(maps));
    const bool ok = make_map(&maps.x, a.x, DV, a.T, a.BH, kGlaTc) && make_map(&maps.y, a.y, DV, a.T, a.BH, kGlaTc) &&
                    make_map(&maps.z, a.z, a.DK, a.T, a.BH, kGlaTc) &&
                    make_map_f32_rows(&maps.g, a.g, a.DK, a.T, a.BH, kGlaTc, 64);
    if (!ok) return fail(CLA_ERR_CUDA, "gla_tc_qk_kernel: tensor map encoding failed");
    return a.rev ? launch_gla_bwd_qk_variant<DV, true>(a, maps, s, grid)
                 : launch_gla_bwd_qk_variant<DV, false>(a, maps, s, grid);
}

template <int DK, bool REV>
int launch_gla_fwd_variant(const GlaArgs &a, const GlaMaps &maps, cudaStream_t s, unsigned int grid) {
    using C = GlaTcCfg<DK>;
    static std::atomic<unsigned long long> smem_set{0};  // per template instance
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(gla_tc_kernel<DK, REV>), C::SMEM);
    if (st) return st;
    gla_tc_kernel<DK, REV><<<grid, kGlaTcThreads, C::SMEM, s>>>(a, maps);
    return check_launch("gla_tc_kernel");
}

template <int DK>
int launch_gla_fwd(const GlaArgs &a, cudaStream_t s, unsigned int grid) {
    GlaMaps maps;
    memset(&maps, 0, sizeof(maps));
    const bool ok = make_map(&maps.q, a.q, DK, a.T, a.BH, kGlaTc) && make_map(&maps.k, a.k, DK, a.T, a.BH, kGlaTc) &&
                    make_map(&maps.v, a.v, a.DV, a.T, a.BH, kGlaTc) &&
                    make_map_f32_rows(&maps.g, a.g, DK, a.T, a.BH, kGlaTc, DK);
    if (!ok) return fail(CLA_ERR_CUDA, "gla_tc_kernel: tensor map encoding failed");
    return a.rev ? launch_gla_fwd_variant<DK, true>(a, maps, s, grid) : launch_gla_fwd_variant<DK, false>(a, maps, s, grid);
}

}  // namespace
}  // namespace cla

using namespace cla;

extern "C" size_t cla_gla_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk) {
    if (!gla_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    return gla_plan(B, H, T, dim_k, dim_v).total;
}

namespace {
int gla_fwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                 const float *S0, float *o, float *ST, float *ckpt, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                 int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    if (B < 0 || H < 0 || T < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!gla_supported(B, H, T, dim_k, dim_v, chunk))
        return fail(CLA_ERR_UNSUPPORTED, "%s: needs dim_k 64 or 128, dim_v a multiple of 64 up to 1024, chunk 64 "
                    "and sizes within one launch (got dim_k %lld, dim_v %lld, chunk %d)", fn, (long long)dim_k,
                    (long long)dim_v, chunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t BH = B * H;
    if (BH == 0) return CLA_OK;
    const size_t sbytes = sizeof(float) * BH * dim_k * dim_v;
    if (T == 0) {
        if (ST) {
            if (S0) CLA_CUDA_TRY(cudaMemcpyAsync(ST, S0, sbytes, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(ST, 0, sbytes, s), fn);
        }
        return CLA_OK;
    }
    if (!q || !k || !v || !log_decay || !o) return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, log_decay, o required", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_decay))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, log_decay must be 16-byte aligned", fn);
    if (!aligned_or_null({o}, 8) || !aligned_or_null({S0, ST}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: o must be 8-byte aligned, S0 and ST 4-byte aligned", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    const GlaPlan pl = gla_plan(B, H, T, dim_k, dim_v);
    if (ws_bytes < pl.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, pl.total);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_alpha, s), fn);
    char *w = static_cast<char *>(ws);
    GlaArgs a;
    memset(&a, 0, sizeof(a));
    a.q = reinterpret_cast<const bf16 *>(q);
    a.k = reinterpret_cast<const bf16 *>(k);
    a.v = reinterpret_cast<const bf16 *>(v);
    a.g = log_decay;
    a.S0 = S0;
    a.o = o;
    a.ST = ST;
    a.rev = 0;
    a.BH = (int)BH;
    a.DV = (int)dim_v;
    a.nzb = pl.nzb;
    a.n_chunks = pl.n_chunks;
    a.seg_chunks = pl.seg_chunks;
    a.n_seg = pl.n_seg;
    a.T = T;
    a.hdr = reinterpret_cast<WsHeader *>(w);
    a.flags = reinterpret_cast<unsigned int *>(w + pl.off_flags);
    a.alpha = reinterpret_cast<float *>(w + pl.off_alpha);
    a.agg = reinterpret_cast<float4 *>(w + pl.off_agg);
    a.incl = reinterpret_cast<float4 *>(w + pl.off_incl);
    a.seg_out = ckpt;  // [n_seg][BH][dim_k][dim_v]: the state entering each segment
    const unsigned int grid = (unsigned int)(pl.units);
    return dim_k == 64 ? launch_gla_fwd<64>(a, s, grid) : launch_gla_fwd<128>(a, s, grid);
}
}  // namespace

extern "C" int cla_gla_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                           const float *S0, float *o, float *ST, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                           int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    return gla_fwd_impl("cla_gla_fwd", q, k, v, log_decay, S0, o, ST, nullptr, B, H, T, dim_k, dim_v, chunk, ws,
                        ws_bytes, stream);
}

extern "C" size_t cla_gla_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk) {
    if (!gla_supported(B, H, T, dim_k, dim_v, chunk) || !gla_bwd_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    const GlaPlan pl = gla_plan(B, H, T, dim_k, dim_v);
    return (size_t)pl.n_seg * (size_t)(B * H) * (size_t)dim_k * (size_t)dim_v * sizeof(float);
}

extern "C" int cla_gla_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                const float *S0, float *o, float *ST, float *ckpt, int64_t B, int64_t H, int64_t T,
                                int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    if (ckpt != nullptr && !aligned16(ckpt))
        return fail(CLA_ERR_INVALID_ARG, "cla_gla_fwd_ckpt: ckpt must be 16-byte aligned");
    if (ckpt != nullptr && !gla_bwd_supported(B, H, T, dim_k, dim_v, chunk))
        return fail(CLA_ERR_UNSUPPORTED, "cla_gla_fwd_ckpt: a checkpoint needs sizes the backward takes "
                    "(dim_k and dim_v 64 or 128)");
    return gla_fwd_impl("cla_gla_fwd_ckpt", q, k, v, log_decay, S0, o, ST, ckpt, B, H, T, dim_k, dim_v, chunk, ws,
                        ws_bytes, stream);
}

extern "C" size_t cla_gla_bwd_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                             int chunk) {
    if (!gla_bwd_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    return gla_bwd_plan(B, H, T, dim_k, dim_v).total;
}

namespace {
int gla_bwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                 const float *S0, const uint16_t *dO, const float *dST, float *dq, float *dk, float *dv,
                 float *dlog_decay, float *dS0, const float *ckpt, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                 int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    if (B < 0 || H < 0 || T < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!gla_bwd_supported(B, H, T, dim_k, dim_v, chunk))
        return fail(CLA_ERR_UNSUPPORTED, "%s: needs dim_k and dim_v 64 or 128, chunk 64 and sizes within one launch "
                    "(got dim_k %lld, dim_v %lld, chunk %d)", fn, (long long)dim_k, (long long)dim_v, chunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t BH = B * H;
    if (BH == 0) return CLA_OK;
    const size_t sbytes = sizeof(float) * BH * dim_k * dim_v;
    if (T == 0) {
        if (dS0) {
            if (dST) CLA_CUDA_TRY(cudaMemcpyAsync(dS0, dST, sbytes, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(dS0, 0, sbytes, s), fn);
        }
        return CLA_OK;
    }
    if (!q || !k || !v || !log_decay || !dO || !dq || !dk || !dv)
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, log_decay, dO, dq, dk, dv required", fn);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(log_decay))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, dO, log_decay must be 16-byte aligned", fn);
    if (!aligned_or_null({dq, dk, dv}, 8) || !aligned_or_null({S0, dST, dlog_decay, dS0}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: dq, dk, dv must be 8-byte aligned, S0, dST, dlog_decay, dS0 4-byte", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    const GlaBwdPlan pl = gla_bwd_plan(B, H, T, dim_k, dim_v);
    if (ws_bytes < pl.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, pl.total);
    char *w = static_cast<char *>(ws);
    float *fs = reinterpret_cast<float *>(w + pl.off_fs);
    const bf16 *Q = reinterpret_cast<const bf16 *>(q), *K = reinterpret_cast<const bf16 *>(k);
    const bf16 *V = reinterpret_cast<const bf16 *>(v), *DO = reinterpret_cast<const bf16 *>(dO);

    auto args_b = [&](int rev) {
        GlaBArgs b;
        memset(&b, 0, sizeof(b));
        b.g = log_decay;
        b.S0 = dST;
        b.rev = rev;
        b.BH = (int)BH;
        b.DK = (int)dim_k;
        b.nzb = (int)(dim_k / 64);
        b.n_chunks = pl.n_chunks;
        b.seg_chunks = pl.seg_chunks;
        b.n_seg = pl.n_seg;
        b.T = T;
        b.hdr = reinterpret_cast<WsHeader *>(w);
        b.flags = reinterpret_cast<unsigned int *>(w + pl.off_flags);
        b.alpha = reinterpret_cast<float *>(w + pl.off_alpha);
        b.agg = reinterpret_cast<float4 *>(w + pl.off_agg);
        b.incl = reinterpret_cast<float4 *>(w + pl.off_incl);
        return b;
    };
    const unsigned int gridB = (unsigned int)((size_t)pl.n_seg * BH * (dim_k / 64));
    int st;
    // dQ: forward traversal, X = dO, Y = V, Z = K, the state from S0; its final state dotted
    // with dST gives the decay gradient's final-state term
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_alpha, s), fn);
    GlaBArgs b = args_b(0);
    b.x = DO;
    b.y = V;
    b.z = K;
    b.S0 = S0;
    b.out = dq;
    b.fs_dot = dST;
    b.fs_part = fs;
    b.seg_in = ckpt;  // the forward's state entering each segment (the same segments), if saved
    st = dim_v == 64 ? launch_gla_bwd_qk<64>(b, s, gridB) : launch_gla_bwd_qk<128>(b, s, gridB);
    if (st) return st;

    // dV and dS0: the forward kernel on the reversed adjoint (q <- k, k <- q, v <- dO, S0 <- dST)
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_alpha, s), fn);
    GlaArgs a;
    memset(&a, 0, sizeof(a));
    a.q = K;
    a.k = Q;
    a.v = DO;
    a.g = log_decay;
    a.S0 = dST;
    a.o = dv;
    a.ST = dS0;
    a.rev = 1;
    a.BH = (int)BH;
    a.DV = (int)dim_v;
    a.nzb = (int)(dim_v / 64);
    a.n_chunks = pl.n_chunks;
    a.seg_chunks = pl.seg_chunks;
    a.n_seg = pl.n_seg;
    a.T = T;
    a.hdr = reinterpret_cast<WsHeader *>(w);
    a.flags = reinterpret_cast<unsigned int *>(w + pl.off_flags);
    a.alpha = reinterpret_cast<float *>(w + pl.off_alpha);
    a.agg = reinterpret_cast<float4 *>(w + pl.off_agg);
    a.incl = reinterpret_cast<float4 *>(w + pl.off_incl);
    // the adjoint state entering each segment, which the dK traversal (same segments, same
    // state) then starts from instead of running its phase 1 and look-back
    a.seg_out = reinterpret_cast<float *>(w + pl.off_seg);
    const unsigned int gridA = (unsigned int)((size_t)pl.n_seg * BH * (dim_v / 64));
    st = dim_k == 64 ? launch_gla_fwd<64>(a, s, gridA) : launch_gla_fwd<128>(a, s, gridA);
    if (st) return st;

    // dK: reversed traversal, X = V, Y = dO, Z = Q, the adjoint state from dST
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_alpha, s), fn);
    b = args_b(1);
    b.x = V;
    b.y = DO;
    b.z = Q;
    b.out = dk;
    b.seg_in = reinterpret_cast<const float *>(w + pl.off_seg);
    st = dim_v == 64 ? launch_gla_bwd_qk<64>(b, s, gridB) : launch_gla_bwd_qk<128>(b, s, gridB);
    if (st) return st;

    if (dlog_decay) {
        float *tsum = reinterpret_cast<float *>(w + pl.off_tsum);
        const unsigned int grid = (unsigned int)((size_t)pl.tiles * BH);
        // 8 key dimensions a thread where the gradients' rows take 16-byte accesses
        const bool vec8 = aligned16(dq) && aligned16(dk) && aligned16(dlog_decay);
        const long long n_units = (long long)pl.tiles * BH;
        const unsigned int grid8 = (unsigned int)((n_units + kGlaDl8Threads / (dim_k / 8) - 1) /
                                                  (kGlaDl8Threads / (dim_k / 8)));
        if (vec8)
            gla_dlog_tile_sums8_kernel<<<grid8, kGlaDl8Threads, 0, s>>>(Q, dq, K, dk, tsum, (int)dim_k, T, pl.tiles,
                                                                       n_units);
        else
            gla_dlog_tile_sums_kernel<<<grid, (unsigned int)dim_k, 0, s>>>(Q, dq, K, dk, tsum, (int)dim_k, T, pl.tiles);
        st = check_launch("gla_dlog_tile_sums_kernel");
        if (st) return st;
        gla_dlog_tile_suffix_kernel<<<(unsigned int)BH, (unsigned int)dim_k, 0, s>>>(tsum, fs, (int)dim_k, pl.tiles);
        st = check_launch("gla_dlog_tile_suffix_kernel");
        if (st) return st;
        if (vec8)
            gla_dlog_finalize8_kernel<<<grid8, kGlaDl8Threads, 0, s>>>(Q, dq, K, dk, tsum, dlog_decay, (int)dim_k, T,
                                                                      pl.tiles, n_units);
        else
            gla_dlog_finalize_kernel<<<grid, (unsigned int)dim_k, 0, s>>>(Q, dq, K, dk, tsum, dlog_decay, (int)dim_k, T,
                                                                          pl.tiles);
        st = check_launch("gla_dlog_finalize_kernel");
    }
    return st;
}
}  // namespace

extern "C" int cla_gla_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                           const float *S0, const uint16_t *dO, const float *dST, float *dq, float *dk, float *dv,
                           float *dlog_decay, float *dS0, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                           int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    return gla_bwd_impl("cla_gla_bwd", q, k, v, log_decay, S0, dO, dST, dq, dk, dv, dlog_decay, dS0, nullptr, B, H,
                        T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}

extern "C" int cla_gla_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                const float *S0, const uint16_t *dO, const float *dST, float *dq, float *dk,
                                float *dv, float *dlog_decay, float *dS0, const float *ckpt, int64_t B, int64_t H,
                                int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                                void *stream) {
    if (ckpt != nullptr && !aligned16(ckpt))
        return fail(CLA_ERR_INVALID_ARG, "cla_gla_bwd_ckpt: ckpt must be 16-byte aligned");
    return gla_bwd_impl("cla_gla_bwd_ckpt", q, k, v, log_decay, S0, dO, dST, dq, dk, dv, dlog_decay, dS0, ckpt, B,
                        H, T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}
