// chunk_la_tc.cuh -- the chunk kernel of chunk_la.cu on Blackwell's fifth-
// generation tensor cores: TMA tile loads, tcgen05.mma with the accumulators
// in tensor memory (TMEM).  Included by chunk_la.cu (shares its
// LaArgs, decay helpers and workspace layout); computes exactly the products
// documented there:
//     P       = X Y^T                     (M = Tc, N = Tc, K = DX)   smem x smem
//     O_inter = X S_hi + X S_lo           (M = Tc, N = 64, K = DX)   smem x smem
//     dS      = Y^T [Zs_hi | Zs_lo]       (M = DX, N = 128, K = Tc)  smem x smem
//     O_intra = P_hi Z + P_lo Z           (M = Tc, N = 64, K = Tc)   tmem x smem
// where Zs = diag(w_state) Z and P is masked and decayed in registers between
// the first and the last product, split into two bf16 parts and written back
// to TMEM as the A operand.  OUT = O_intra + diag(w_out) O_inter, State =
// alpha State + (dS_hi + dS_lo), the two 64-column halves of the dS product.  A value x split into bf16 parts is x = hi + lo + e with
// |e| < 2^-16 |x| (both parts by truncation, see split_bf16x2).
//
// Warp roles.  Warp 8 (the producer) issues every TMA load and every MMA
// (warp-wide, under elect.sync), so the tensor pipe works ahead of the
// elementwise stages (the next chunk's P is formed while this chunk's output
// is written).  Warp 9 computes the decays of each chunk one visit ahead.
// Warps 0..7 (the math warps) do the elementwise work: Zs, masking, the State
// recurrence and the output epilogue, staged in shared memory and written by
// one TMA store per warp.  They hand work to the producer through named
// barriers and learn of finished MMAs and loads through mbarriers.  A math
// warp w reads TMEM lane quarter w & 3 (the lanes a warp may access are fixed
// by its rank within its warpgroup); warps w and w + 4 split the columns.
// The thread whose lane holds row r of an M-row accumulator owns that row
// (M = 128: lane = row; M = 64: rows 16q..16q+15 sit in lanes 32q..32q+15).
//
// Operand layouts in shared memory use the 128-byte swizzle (8 rows of 128
// bytes per 1024-byte atom, 16-byte chunks XOR-ed with the row's low 3 bits),
// as TMA writes them: X, Y as K-major A/B operands (blocks of 64 columns),
// Y as the MN-major A operand of dS, Z and S as MN-major B operands, Zs as
// a K-major B operand written by the threads.
//
// A block covers one segment of chunks of one (batch, head) and 64 output
// columns.  Phase 1 sums the segment's state from zero; a decoupled look-back
// over the segments before it gives its incoming state; phase 2 runs the
// chunks from that state and writes the outputs.  With LaArgs::seg_out the
// incoming state is also saved; with LaArgs::seg_in it is read from there
// (possibly transposed: another traversal's state) and phase 1 and the
// look-back are skipped.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_ptx.cuh"

namespace cla {
namespace {

// ----------------------------------------------------------------- configuration
template <int DX, int TC>
struct TcCfg {
    static constexpr int NT = 320;  // 8 math warps (w and w + 4 share TMEM lane quarter w), producer, decay warp
    static constexpr int KBX = DX / 64;  // 64-column blocks of X and Y
    static constexpr int KBT = TC / 64;  // 64-token blocks of Zs
    // Compact layout (DX = Tc = 64, whose every stage is short): two blocks per SM, so one
    // block's tensor-core and barrier latencies overlap the other's work.  It needs half the
    // TMEM (256 columns): the scores are masked in place, and dS accumulates Y^T Zs_hi and
    // Y^T Zs_lo in one 64-column accumulator (two N = 64 products instead of one N = 128).
    static constexpr bool COMPACT = (DX == 64 && TC == 64);
    static constexpr int MIN_BLOCKS = COMPACT ? 2 : 1;
    // TMEM columns: P (fp32), the accumulators, and the masked P as bf16 parts.
    static constexpr uint32_t C_P = 0;
    static constexpr uint32_t C_OI = TC;        // O_inter
    static constexpr uint32_t C_OA = TC + 64;   // O_intra
    // dS: Y^T Zs_hi in 64 columns, then Y^T Zs_lo in 64 (compact: both in the same 64)
    static constexpr uint32_t C_DS = TC + 128;
    // masked, decayed P as the bf16 A operand of O_intra: per 32-token piece,
    // the high part in its first 16 columns and the low part in the next 16
    static constexpr uint32_t C_PB = COMPACT ? C_P : TC + 256;
    static constexpr uint32_t TMEM_COLS = COMPACT ? 256 : 512;
    static_assert(COMPACT ? (C_DS + 64 <= TMEM_COLS) : (C_PB + TC <= TMEM_COLS), "tensor memory budget");
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int X_BYTES = KBX * TC * 128;
    static constexpr int Z_BYTES = TC * 128;
    static constexpr int S_BYTES = DX * 128;         // one bf16 part of State (MN-major)
    // Zs as the K-major B operand of dS, N = 128: per 64-token block, rows
    // 0..63 hold Zs_hi and rows 64..127 Zs_lo (16 KB per block)
    static constexpr int ZS_BYTES = KBT * 128 * 128;
    static constexpr int DEC_STRIDE = 5 * TC + 4;  // floats per decay buffer (below)
    static constexpr int DEC_BYTES = (2 * DEC_STRIDE + 2 * TC) * 4;
    // X is double-buffered where shared memory allows (every shape but DX = Tc = 128), so
    // the next chunk's X load overlaps this chunk instead of waiting for its O_inter
    static constexpr int SMEM_ONE_X = 3 * X_BYTES + 3 * Z_BYTES + 2 * S_BYTES + ZS_BYTES + DEC_BYTES + 128 + 1024;
    static constexpr bool XDB = SMEM_ONE_X + X_BYTES <= 227 * 1024;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_X1 = XDB ? X_BYTES : 0;
    static constexpr int OFF_Y0 = OFF_X + (XDB ? 2 : 1) * X_BYTES;
    static constexpr int OFF_Y1 = OFF_Y0 + X_BYTES;
    static constexpr int OFF_Z0 = OFF_Y1 + X_BYTES;
    static constexpr int OFF_Z1 = OFF_Z0 + Z_BYTES;
    static constexpr int OFF_W = OFF_Z1 + Z_BYTES;
    static constexpr int OFF_SH = OFF_W + Z_BYTES;
    static constexpr int OFF_SL = OFF_SH + S_BYTES;
    // Zs; after the chunk's dS product, the fp32 output tile (two
    // 128-byte-swizzled halves of Tc rows x 32 columns) for the TMA store
    static constexpr int OFF_ZS = OFF_SL + S_BYTES;
    static constexpr int OFF_DEC = OFF_ZS + ZS_BYTES;
    // decays, two buffers (chunk sequence number parity) of cl, zr, w_out,
    // w_state, g [Tc] and alpha; then the two half-row dot products [2][Tc]
    static constexpr int OFF_BAR = OFF_DEC + DEC_BYTES;
    static constexpr int SMEM = OFF_BAR + 128 + 1024;  // 13 mbarriers + alignment slack
    static_assert(SMEM == SMEM_ONE_X + (XDB ? X_BYTES : 0), "shared memory layout");
    static_assert(ZS_BYTES == TC * 64 * 4, "the output tile fits the Zs buffer");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct TcMaps {
    CUtensorMap x, y, z, w, out;
};

// Named barriers between the 8 math warps and the producer warp.
constexpr int kBarMath = 1;   // the 256 math threads
constexpr int kBarZs = 2;     // math: Zs written          -> producer may issue dS
constexpr int kBarPmask = 3;  // math: P masked and split  -> producer may issue O_intra
constexpr int kBarDone = 4;   // math: chunk finished      -> producer may issue the next O_inter
constexpr int kMathThreads = 256;
constexpr int kAllThreads = 288;    // math warps + producer: the named-barrier count
constexpr int kBlockThreads = 320;  // + the decay warp

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int DX, int TC, bool REV>
__global__ void __launch_bounds__(kBlockThreads, TcCfg<DX, TC>::MIN_BLOCKS)
    la_tc_kernel(const __grid_constant__ TcMaps maps, const LaArgs p) {
    using C = TcCfg<DX, TC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    __shared__ uint32_t s_tmem;
    __shared__ unsigned int s_ticket, s_flag;
    __shared__ float s_palpha;
    __shared__ float s_red[8];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = (warp == 8);
    // mbarriers: 0 X (buffer 0), 1 YZ0, 2 YZ1, 3 W, 4 P, 5 dS, 6 O_intra, 7 O_inter, 8-9 decay
    // buffers full (the decay warp's 32 lanes arrive), 10-11 decay buffers empty (one arrival per
    // math warp), 12 X buffer 1
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    // TMEM first (before taking a ticket, so every ticket holder owns its TMEM)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
    }
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(12), 1);
        mbar_init(bar(8), 32);
        mbar_init(bar(9), 32);
        mbar_init(bar(10), 8);
        mbar_init(bar(11), 8);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_ticket = atomicAdd(&p.hdr->ticket[p.ticket_slot], 1u);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const unsigned int tk = s_ticket;
    const int per_seg = p.BH * p.nzb;
    const int sidx = (int)(tk / per_seg);
    const int bh = (int)(tk % per_seg) / p.nzb;
    const int zb = (int)(tk % per_seg) % p.nzb;
    const int seg = REV ? (p.n_seg - 1 - sidx) : sidx;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
    const int nc = c_end - c_begin;
    const size_t unit = ((size_t)seg * p.BH + bh) * p.nzb + zb;
    auto chunk_at = [&](int i) { return REV ? (c_end - 1 - i) : (c_begin + i); };
    const bool has_w = p.W != nullptr;
    // With the segments' incoming states given (seg_in), phase 1 and the look-back are
    // skipped: the chunk visits are those of phase 2 only, nc..2nc-1, and v0 is the first.
    const bool skip1 = p.seg_in != nullptr;
    const int v0 = skip1 ? nc : 0;
    bool timed_out = false;
    uint32_t ph = 0u;  // bit i: the phase parity mbarrier i completes next (a register, not an array)
    auto wait = [&](int i) {
        if (!mbar_wait(bar(i), (ph >> i) & 1u)) timed_out = true;
        ph ^= 1u << i;
    };
    // Decays are computed once per chunk visit, by the decay warp.  Visits are
    // numbered 0..2nc-1 (phase 1, then phase 2); visit n uses decay buffer
    // n & 1, whose full and empty mbarriers complete one phase per use: visit
    // n is use n >> 1 of its buffer.
    float *dec = reinterpret_cast<float *>(smem + C::OFF_DEC);
    auto dbuf = [&](int n) { return dec + ((n - v0) & 1) * C::DEC_STRIDE; };
    float *dotp = dec + 2 * C::DEC_STRIDE;  // [2][Tc] half-row dot products

    if (producer) {
        // ============================================================ producer warp
        const bool leader = (lane == 0);
        // X buffer xb (always 0 without double buffering) and its full barrier
        auto xbar = [&](int xb) { return xb ? 12 : 0; };
        auto issue_x = [&](int xb, int chunk) {
            const uint32_t bx = bar(xbar(xb));
            mbar_expect_tx(bx, (uint32_t)C::X_BYTES);
            for (int kb = 0; kb < C::KBX; ++kb)
                tma_load_3d(sbase + (xb ? C::OFF_X1 : C::OFF_X) + kb * TC * 128, &maps.x, kb * 64, chunk * TC, bh, bx);
        };
        auto issue_yz = [&](int b, int chunk) {
            mbar_expect_tx(bar(1 + b), (uint32_t)(C::X_BYTES + C::Z_BYTES));
            const uint32_t oy = b ? C::OFF_Y1 : C::OFF_Y0, oz = b ? C::OFF_Z1 : C::OFF_Z0;
            for (int kb = 0; kb < C::KBX; ++kb)
                tma_load_3d(sbase + oy + kb * TC * 128, &maps.y, kb * 64, chunk * TC, bh, bar(1 + b));
            tma_load_3d(sbase + oz, &maps.z, zb * 64, chunk * TC, bh, bar(1 + b));
        };
        auto issue_w = [&](int chunk) {
            mbar_expect_tx(bar(3), (uint32_t)C::Z_BYTES);
            tma_load_3d(sbase + C::OFF_W, &maps.w, zb * 64, chunk * TC, bh, bar(3));
        };
        // Descriptors of every operand tile, built once; a K step adds a constant
        // byte offset (>> 4) to the start-address field.
        const uint64_t dX0 = smem_desc(sbase + C::OFF_X, 16, 1024);                 // K-major
        auto dX = [&](int xb) { return dX0 + (uint64_t)(xb * ((C::OFF_X1 - C::OFF_X) >> 4)); };
        // The two Y and Z buffers differ only in their start address: buffer b's descriptor is
        // buffer 0's plus b times the buffer size (no arrays indexed at run time: those would
        // live in local memory, a cache miss in front of an MMA issue).
        const uint64_t dY0 = smem_desc(sbase + C::OFF_Y0, 16, 1024);                 // K-major
        const uint64_t dYt0 = smem_desc(sbase + C::OFF_Y0, TC * 128, 1024);          // MN-major (Y^T)
        const uint64_t dZ0 = smem_desc(sbase + C::OFF_Z0, 8192, 1024);               // MN-major
        static_assert(C::OFF_Y1 - C::OFF_Y0 == C::X_BYTES && C::OFF_Z1 - C::OFF_Z0 == C::Z_BYTES, "buffer pairs");
        auto dY = [&](int b) { return dY0 + (uint64_t)(b * (C::X_BYTES >> 4)); };
        auto dYt = [&](int b) { return dYt0 + (uint64_t)(b * (C::X_BYTES >> 4)); };
        auto dZ = [&](int b) { return dZ0 + (uint64_t)(b * (C::Z_BYTES >> 4)); };
        const uint64_t dS[2] = {smem_desc(sbase + C::OFF_SH, 8192, 1024), smem_desc(sbase + C::OFF_SL, 8192, 1024)};
        const uint64_t dZs = smem_desc(sbase + C::OFF_ZS, 16, 1024);               // K-major, 128 rows
        auto issue_state_mma = [&](int b) {
            const uint64_t a0 = dYt(b);
            if constexpr (C::COMPACT) {
                // dS = Y^T Zs_hi + Y^T Zs_lo in one accumulator (M = DX, N = 64, K = Tc, twice)
                constexpr uint32_t id = idesc_bf16(DX, 64, 1, 0);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < TC / 16; ++kk)
                        mma_ss_w(tmem + C::C_DS, a0 + (uint64_t)(kk * 2048 / 16),
                                 dZs + (uint64_t)(((kk >> 2) * 128 * 128 + (kk & 3) * 32 + part * 64 * 128) / 16), id,
                                 (part | kk) ? 1u : 0u);
            } else {
                // dS = Y^T [Zs_hi | Zs_lo]  (M = DX, N = 128, K = Tc)
                constexpr uint32_t id = idesc_bf16(DX, 128, 1, 0);
#pragma unroll
                for (int kk = 0; kk < TC / 16; ++kk)
                    mma_ss_w(tmem + C::C_DS, a0 + (uint64_t)(kk * 2048 / 16),
                             dZs + (uint64_t)(((kk >> 2) * 128 * 128 + (kk & 3) * 32) / 16), id, kk ? 1u : 0u);
            }
        };
        auto issue_p = [&](int b, int xb) {
            constexpr uint32_t idp = idesc_bf16(TC, TC, 0, 0);
            const uint64_t b0 = dY(b), a0 = dX(xb);
#pragma unroll
            for (int kk = 0; kk < DX / 16; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * TC * 128 + (kk & 3) * 32) / 16);
                mma_ss_w(tmem + C::C_P, a0 + off, b0 + off, idp, kk ? 1u : 0u);
            }
        };
        auto issue_inter = [&](int xb) {
            constexpr uint32_t ido = idesc_bf16(TC, 64, 0, 1);
            const uint64_t a0 = dX(xb);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
                for (int kk = 0; kk < DX / 16; ++kk)
                    mma_ss_w(tmem + C::C_OI, a0 + (uint64_t)(((kk >> 2) * TC * 128 + (kk & 3) * 32) / 16),
                             dS[part] + (uint64_t)(kk * 2048 / 16), ido, (part | kk) ? 1u : 0u);
            }
        };
        auto issue_intra = [&](int b) {
            constexpr uint32_t id = idesc_bf16(TC, 64, 0, 1);
            const uint64_t b0 = dZ(b);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
                for (int kk = 0; kk < TC / 16; ++kk) {
                    // tokens 16kk.. lie in piece kk/2: high part at its columns 0..15, low part at 16..31
                    const uint32_t acol = C::C_PB + (uint32_t)(kk >> 1) * 32 + part * 16 + (kk & 1) * 8;
                    mma_ts_w(tmem + C::C_OA, tmem + acol, b0 + (uint64_t)(kk * 2048 / 16), id, (part | kk) ? 1u : 0u);
                }
            }
        };
        // ---- phase 1: dS per chunk
        if (leader && !skip1) {
            issue_yz(0, chunk_at(0));
            if (nc > 1) issue_yz(1, chunk_at(1));
        }
        for (int i = 0; i < (skip1 ? 0 : nc); ++i) {
            const int b = i & 1;
            wait(1 + b);
            bar_sync(kBarZs, kAllThreads);
            tc_fence_after();
            issue_state_mma(b);
            mma_commit_w(bar(5));
            wait(5);
            if (leader && i + 2 < nc) issue_yz(b, chunk_at(i + 2));
        }
        // ---- phase 2 loads and the first scores while the math warps look back
        // (chunk i's X sits in buffer i & 1 with double buffering, else in buffer 0)
        auto xbuf = [&](int i) { return C::XDB ? (i & 1) : 0; };
        if (leader) {
            issue_yz(0, chunk_at(0));
            if (nc > 1) issue_yz(1, chunk_at(1));
            issue_x(0, chunk_at(0));
            if (C::XDB && nc > 1) issue_x(1, chunk_at(1));
            if (has_w) issue_w(chunk_at(0));
        }
        wait(1);
        wait(xbar(0));
        tc_fence_after();
        issue_p(0, 0);
        mma_commit_w(bar(4));
        for (int i = 0; i < nc; ++i) {
            const int b = i & 1;
            bar_sync(kBarDone, kAllThreads);  // previous chunk finished; State's bf16 parts written
            tc_fence_after();
            issue_inter(xbuf(i));
            mma_commit_w(bar(7));
            if (leader && has_w && i > 0) issue_w(chunk_at(i));
            __syncwarp();
            bar_sync(kBarZs, kAllThreads);
            tc_fence_after();
            issue_state_mma(b);
            mma_commit_w(bar(5));
            wait(7);  // P and O_inter done: chunk i's X buffer is free
            if (leader) {
                if (C::XDB) {
                    if (i + 2 < nc) issue_x(b, chunk_at(i + 2));
                } else if (i + 1 < nc) {
                    issue_x(0, chunk_at(i + 1));
                }
            }
            bar_sync(kBarPmask, kAllThreads);  // masked P written, P read
            tc_fence_after();
            issue_intra(b);
            mma_commit_w(bar(6));
            // compact: the next P overwrites the masked scores O_intra reads
            if (C::COMPACT) wait(6);
            if (i + 1 < nc) {
                wait(1 + (b ^ 1));
                wait(xbar(xbuf(i + 1)));
                tc_fence_after();
                issue_p(b ^ 1, xbuf(i + 1));
                mma_commit_w(bar(4));
            }
            if (!C::COMPACT) wait(6);
            wait(5);
            if (leader && i + 2 < nc) issue_yz(b, chunk_at(i + 2));
        }
        bar_sync(kBarDone, kAllThreads);  // the last chunk's arrival
    } else if (warp == 9) {
        // ============================================================ decay warp
        const float *Lb = p.ell + (size_t)bh * p.T;
        // decays of visit n, by the whole warp: cl_r = in-chunk sum of log2 a up to r (resets
        // skipped), zr_r = last reset at or before r, w_out / w_state, the column factors g of
        // the off-diagonal score pieces, and alpha = the chunk's total decay
        constexpr int PER = TC / 32;
        float ell_pre[PER];  // log-decays of the next visit, loaded one visit ahead
        auto load_ell = [&](int n) {
            const long long t0 = (long long)chunk_at(n < nc ? n : n - nc) * TC;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const long long t = t0 + lane * PER + k;
                ell_pre[k] = (t < p.T) ? __ldg(Lb + t) : 0.f;
            }
        };
        auto compute_decays = [&](int n) {
            float *cl = dbuf(n);
            int *zr = reinterpret_cast<int *>(cl + TC);
            float *wout = cl + 2 * TC, *wst = cl + 3 * TC, *gcol = cl + 4 * TC;
            float v[PER];
            int zz[PER];
            float run = 0.f;
            int lastz = -1;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int r = lane * PER + k;
                const float l = ell_pre[k];
                const bool reset = (l == -INFINITY);
                run += reset ? 0.f : l * kLog2e;
                if (reset) lastz = r;
                v[k] = run;
                zz[k] = lastz;
            }
            float tot = run;
            int zt = lastz;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, tot, off);
                const int oz = __shfl_up_sync(0xffffffffu, zt, off);
                if (lane >= off) {
                    tot += o;
                    zt = max(zt, oz);
                }
            }
            float ex = __shfl_up_sync(0xffffffffu, tot, 1);
            int zex = __shfl_up_sync(0xffffffffu, zt, 1);
            if (lane == 0) {
                ex = 0.f;
                zex = -1;
            }
            const float cL = __shfl_sync(0xffffffffu, tot, 31);
            const int zL = __shfl_sync(0xffffffffu, zt, 31);
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                v[k] += ex;
                zz[k] = max(zz[k], zex);
                cl[lane * PER + k] = v[k];
                zr[lane * PER + k] = zz[k];
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int r = lane * PER + k;
                const float lam = zz[k] >= 0 ? 0.f : ex2(v[k]);
                const float gam = zL > r ? 0.f : ex2(cL - v[k]);
                wout[r] = REV ? gam : lam;
                wst[r] = REV ? lam : gam;
                // D_rs = 2^(cl_r - cl_s) over a 32-token piece of s that row r lies past
                // (forward: every s < r; reversed: every s > r) splits as
                // 2^(cl_r - cl_e) * 2^(cl_e - cl_s), e the piece's token nearest r.
                // With log-decays <= 0, cl is nonincreasing and both factors are <= 1.
                gcol[r] = REV ? ex2(v[k] - cl[r & ~31]) : ex2(cl[r | 31] - v[k]);
            }
            if (lane == 0) cl[5 * TC] = zL >= 0 ? 0.f : ex2(cL);
            mbar_arrive(bar(8 + ((n - v0) & 1)));  // all 32 lanes: release of this lane's writes
        };
        load_ell(v0);
        for (int n = v0; n < 2 * nc; ++n) {
            const int use = (n - v0) >> 1;
            if (use > 0 && !mbar_wait(bar(10 + ((n - v0) & 1)), (uint32_t)((use - 1) & 1))) timed_out = true;
            compute_decays(n);
            if (n + 1 < 2 * nc) load_ell(n + 1);
        }
    } else {
        // ============================================================ math warps
        const int q = warp & 3;    // TMEM lane quarter
        const int hf = warp >> 2;  // which half of the columns this warp handles
        const int mtid = tid;      // 0..255
        // This thread's row and columns.  An accumulator of 128 rows keeps row m in TMEM lane m:
        // a thread holds its lane's row, 32 columns (this warp's half of 64).  One of 64 rows keeps
        // rows 16q..16q+15 in lanes 32q..32q+15: both halves of the warp read those lanes, threads
        // 16..31 taking the upper 16 of the warp's 32 columns.  Token rows (scores, outputs) have
        // T_c rows, state rows (dS, State) DX.
        constexpr int OW = (TC == 128) ? 32 : 16;  // output columns per thread
        constexpr int SW = (DX == 128) ? 32 : 16;  // state columns per thread
        const int prow = (TC == 128) ? q * 32 + lane : q * 16 + (lane & 15);
        const int srow = (DX == 128) ? q * 32 + lane : q * 16 + (lane & 15);
        const int ocol = hf * 32 + ((TC == 128) ? 0 : (lane >> 4) * 16);  // of the 64 output columns
        const int scol = hf * 32 + ((DX == 128) ? 0 : (lane >> 4) * 16);  // of the 64 state columns
        const uint32_t tlane = (uint32_t)(q * 32) << 16;
        auto wait_dec = [&](int n) {
            if (!mbar_wait(bar(8 + ((n - v0) & 1)), (uint32_t)(((n - v0) >> 1) & 1))) timed_out = true;
        };

        // Zs = diag(w_state) Z as two bf16 parts, K-major [64 rows n][Tc tokens]: 8x8 blocks of
        // Z read transposed (ldmatrix.trans), scaled per token, split, written with stmatrix.
        auto write_zs = [&](int b, const float *wst) {
            const uint32_t zt = sbase + (b ? C::OFF_Z1 : C::OFF_Z0);
            constexpr int NBLK = (TC / 8) * 8;
            const int j = lane & 7, blk_in = lane >> 3;
#pragma unroll
            for (int it = 0; it < NBLK / 32; ++it) {
                const int g4 = warp + 8 * it;
                const int tb = g4 >> 1;
                uint32_t r[4];
                ldsm_x4_trans(zt + sw128(tb * 8 + j, (4 * (g4 & 1) + blk_in) * 8), r);
                const int t = tb * 8 + 2 * (lane & 3);
                const float2 w2 = *reinterpret_cast<const float2 *>(wst + t);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    split_bf16x2(__fmul2_rn(unpack_bf16(r[i]), w2), hi[i], lo[i]);
                }
                const int nrow = (4 * (g4 & 1) + blk_in) * 8 + j;
                const uint32_t off = (uint32_t)((tb * 8) >> 6) * 128 * 128 + sw128(nrow, (tb * 8) & 63);
                stsm_x4(sbase + C::OFF_ZS + off, hi);
                stsm_x4(sbase + C::OFF_ZS + off + 64 * 128, lo);
            }
        };
        float S[SW];
#pragma unroll
        for (int c = 0; c < SW; ++c) S[c] = 0.f;
        auto state_accumulate = [&](float alpha) {
            if constexpr (C::COMPACT) {  // both bf16 parts of Zs already summed in one accumulator
                uint32_t rd[SW];
                tmem_ld_cols<SW>(tmem + tlane + C::C_DS + hf * 32, rd);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < SW / 2; ++jj) {
                    const float2 v = __ffma2_rn(make_float2(alpha, alpha), make_float2(S[2 * jj], S[2 * jj + 1]),
                                                make_float2(__uint_as_float(rd[2 * jj]), __uint_as_float(rd[2 * jj + 1])));
                    S[2 * jj] = v.x;
                    S[2 * jj + 1] = v.y;
                }
                return;
            }
            uint32_t rh[SW], rl[SW];
            tmem_ld_cols<SW>(tmem + tlane + C::C_DS + hf * 32, rh);
            tmem_ld_cols<SW>(tmem + tlane + C::C_DS + 64 + hf * 32, rl);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < SW / 2; ++jj) {
                const float2 d = __fadd2_rn(make_float2(__uint_as_float(rh[2 * jj]), __uint_as_float(rh[2 * jj + 1])),
                                            make_float2(__uint_as_float(rl[2 * jj]), __uint_as_float(rl[2 * jj + 1])));
                const float2 v = __ffma2_rn(make_float2(alpha, alpha), make_float2(S[2 * jj], S[2 * jj + 1]), d);
                S[2 * jj] = v.x;
                S[2 * jj + 1] = v.y;
            }
        };
        auto write_s_smem = [&]() {
#pragma unroll
            for (int c = 0; c < SW / 8; ++c) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    split_bf16x2(make_float2(S[c * 8 + 2 * h], S[c * 8 + 2 * h + 1]), hi[h], lo[h]);
                }
                const uint32_t off = sw128(srow, scol + c * 8);
                *reinterpret_cast<uint4 *>(smem + C::OFF_SH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + C::OFF_SL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        };

        // ---- phase 1
        float alpha_seg = 1.f;
        for (int i = 0; i < (skip1 ? 0 : nc); ++i) {
            const int b = i & 1;
            wait(1 + b);
            wait_dec(i);
            const float *dv = dbuf(i);
            const float alpha = dv[5 * TC];
            alpha_seg *= alpha;
            write_zs(b, dv + 3 * TC);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(10 + (i & 1)));  // this warp is done with visit i's decays
            fence_async_smem();
            bar_arrive(kBarZs, kAllThreads);
            wait(5);
            tc_fence_after();
            state_accumulate(alpha);
            tc_fence_before();
        }

        // ---- look-back
        const bool first = REV ? (seg == p.n_seg - 1) : (seg == 0);
        float4 *agg4 = p.agg + unit * (size_t)(DX * 16);
        float4 *inc4 = p.incl + unit * (size_t)(DX * 16);
        auto load_state0 = [&](float (&dst)[SW], float scale, bool add) {
            float v[SW];
            const int col0 = zb * 64 + scol;
            if (p.state0 == nullptr) {
#pragma unroll
                for (int c = 0; c < SW; ++c) v[c] = 0.f;
            } else if (p.trans0) {  // [DZ][DX]: lanes read consecutive rows
#pragma unroll
                for (int c = 0; c < SW; ++c) v[c] = __ldg(p.state0 + ((size_t)bh * p.DZ + col0 + c) * DX + srow);
            } else {  // [DX][DZ]: this thread's columns are contiguous
                const float *src = p.state0 + ((size_t)bh * DX + srow) * p.DZ + col0;
                if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
                    for (int c4 = 0; c4 < SW / 4; ++c4) {
                        const float4 f = __ldg(reinterpret_cast<const float4 *>(src) + c4);
                        v[4 * c4] = f.x;
                        v[4 * c4 + 1] = f.y;
                        v[4 * c4 + 2] = f.z;
                        v[4 * c4 + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < SW; ++c) v[c] = __ldg(src + c);
                }
            }
#pragma unroll
            for (int c = 0; c < SW; ++c) dst[c] = add ? fmaf(scale, v[c], dst[c]) : v[c];
        };
        // look-back payloads are [column / 4][row] float4s; this thread's columns start at scol
        float Sin[SW];
#pragma unroll
        for (int c = 0; c < SW; ++c) Sin[c] = 0.f;
        // a segment's incoming state in [n_seg][BH][rows][cols] (seg_trans = 0) or with rows and
        // columns swapped (seg_trans = 1)
        const size_t seg_base = ((size_t)seg * p.BH + bh) * (size_t)DX * p.DZ;
        if (skip1) {
            const int col0 = zb * 64 + scol;
            if (p.seg_trans) {  // lanes read consecutive rows
#pragma unroll
                for (int c = 0; c < SW; ++c) Sin[c] = __ldg(p.seg_in + seg_base + (size_t)(col0 + c) * DX + srow);
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(p.seg_in + seg_base + (size_t)srow * p.DZ + col0);
#pragma unroll
                for (int c4 = 0; c4 < SW / 4; ++c4) {
                    const float4 f = __ldg(src + c4);
                    Sin[4 * c4] = f.x;
                    Sin[4 * c4 + 1] = f.y;
                    Sin[4 * c4 + 2] = f.z;
                    Sin[4 * c4 + 3] = f.w;
                }
            }
        } else if (first) {
            load_state0(Sin, 1.f, false);
        } else {
#pragma unroll
            for (int c4 = 0; c4 < SW / 4; ++c4)
                __stcg(agg4 + (scol / 4 + c4) * DX + srow,
                       make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]));
            if (mtid == 0) p.alpha_ws[unit] = alpha_seg;
            bar_sync(kBarMath, kMathThreads);
            // the barrier orders every math thread's stores before thread 0's fence (cumulativity)
            if (mtid == 0) {
                __threadfence();
                st_release(p.flags + unit, 1u);
            }
            float accA = 1.f;
            int j = REV ? seg + 1 : seg - 1;
            while (true) {
                const size_t up = ((size_t)j * p.BH + bh) * p.nzb + zb;
                if (mtid == 0) {
                    const unsigned int f = wait_flag(p.flags + up, p.hdr, 30u + (unsigned)p.ticket_slot);
                    s_flag = f;
                    if (f == 1u) s_palpha = ld_cg(p.alpha_ws + up);
                }
                bar_sync(kBarMath, kMathThreads);
                const unsigned int f = s_flag;
                const float pa = s_palpha;
                bar_sync(kBarMath, kMathThreads);
                if (f == 2u || f == 1u) {
                    const float4 *src = (f == 2u ? p.incl : p.agg) + up * (size_t)(DX * 16);
#pragma unroll
                    for (int c4 = 0; c4 < SW / 4; ++c4) {
                        const float4 v = ld_cg4(src + (scol / 4 + c4) * DX + srow);
                        Sin[4 * c4] = fmaf(accA, v.x, Sin[4 * c4]);
                        Sin[4 * c4 + 1] = fmaf(accA, v.y, Sin[4 * c4 + 1]);
                        Sin[4 * c4 + 2] = fmaf(accA, v.z, Sin[4 * c4 + 2]);
                        Sin[4 * c4 + 3] = fmaf(accA, v.w, Sin[4 * c4 + 3]);
                    }
                    if (f == 2u) break;
                    accA *= pa;
                    j = REV ? j + 1 : j - 1;
                    if (j < 0 || j >= p.n_seg) {
                        load_state0(Sin, accA, true);
                        break;
                    }
                } else {
                    break;
                }
            }
        }
        if (!skip1) {
#pragma unroll
            for (int c4 = 0; c4 < SW / 4; ++c4)
                __stcg(inc4 + (scol / 4 + c4) * DX + srow,
                       make_float4(fmaf(alpha_seg, Sin[4 * c4], S[4 * c4]), fmaf(alpha_seg, Sin[4 * c4 + 1], S[4 * c4 + 1]),
                                   fmaf(alpha_seg, Sin[4 * c4 + 2], S[4 * c4 + 2]),
                                   fmaf(alpha_seg, Sin[4 * c4 + 3], S[4 * c4 + 3])));
            bar_sync(kBarMath, kMathThreads);
            if (mtid == 0) {
                __threadfence();
                st_release(p.flags + unit, 2u);
            }
            if (p.seg_out != nullptr) {  // this segment's incoming state, for a later traversal
                float4 *dst = reinterpret_cast<float4 *>(p.seg_out + seg_base + (size_t)srow * p.DZ + zb * 64 + scol);
#pragma unroll
                for (int c4 = 0; c4 < SW / 4; ++c4)
                    dst[c4] = make_float4(Sin[4 * c4], Sin[4 * c4 + 1], Sin[4 * c4 + 2], Sin[4 * c4 + 3]);
            }
        }

        // ---- phase 2
        // the 32-token piece holding this warp's rows; other pieces are either fully masked
        // (the same ones for every chunk: their bf16 parts are zeroed here, once) or lie
        // entirely on the unmasked side of every row (off-diagonal)
        const int rpiece = ((TC == 128) ? q * 32 : q * 16) >> 5;
        constexpr int PIECES = TC / 64;  // pieces of 32 tokens per warp
        auto piece_masked = [&](int piece) { return REV ? (piece < rpiece) : (piece > rpiece); };
        {
            const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int pc = 0; pc < PIECES; ++pc) {
                const int piece = hf * PIECES + pc;
                if (piece_masked(piece)) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) tmem_st8(tmem + tlane + C::C_PB + (uint32_t)(piece * 32 + 8 * c8), zero);
                }
            }
            tmem_st_wait();
        }
#pragma unroll
        for (int c = 0; c < SW; ++c) S[c] = Sin[c];
        write_s_smem();
        fence_async_smem();
        tc_fence_before();
        bar_arrive(kBarDone, kAllThreads);  // State's bf16 parts for chunk 0
        for (int i = 0; i < nc; ++i) {
            const int b = i & 1;
            const long long t0 = (long long)chunk_at(i) * TC;
            const float *cl = dbuf(nc + i);
            const int *zr = reinterpret_cast<const int *>(cl + TC);
            const float *wout = cl + 2 * TC, *wst = cl + 3 * TC, *gcol = cl + 4 * TC;
            wait(1 + b);
            wait_dec(nc + i);
            const float alpha = cl[5 * TC];
            if (lane == 0) tma_store_wait_read();  // this warp's rows of the previous output tile were read
            bar_sync(kBarMath, kMathThreads);
            write_zs(b, wst);
            fence_async_smem();
            bar_arrive(kBarZs, kAllThreads);
            // ---- mask and decay P (fp32, TMEM) into its bf16 parts (TMEM)
            wait(4);
            tc_fence_after();
            {
                const int r = prow;
                const float clr = cl[r];
                const int zrr = zr[r];
                // Masks and decays 16 consecutive tokens tok0.. of a piece for row r (scores p16) and
                // splits the results into bf16x2 parts.  Off-diagonal pieces take the row factor f
                // times the column factors g; without a reset between the piece and the row (zr is
                // nondecreasing) every product is kept (all_keep).  Half a piece at a time keeps the
                // live registers low enough for the compiler to overlap the pairs.
                auto mask16 = [&](const uint32_t(&p16)[16], int piece, int tok0, float f, bool all_keep,
                                  uint32_t(&hi)[8], uint32_t(&lo)[8]) {
                    float cs[16];
                    int zs[16];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {  // 16-byte broadcast loads (same address in every lane)
                        const float4 g = *reinterpret_cast<const float4 *>((piece != rpiece ? gcol : cl) + tok0 + 4 * c4);
                        cs[4 * c4] = g.x;
                        cs[4 * c4 + 1] = g.y;
                        cs[4 * c4 + 2] = g.z;
                        cs[4 * c4 + 3] = g.w;
                        if (REV) {
                            const int4 zv = *reinterpret_cast<const int4 *>(zr + tok0 + 4 * c4);
                            zs[4 * c4] = zv.x;
                            zs[4 * c4 + 1] = zv.y;
                            zs[4 * c4 + 2] = zv.z;
                            zs[4 * c4 + 3] = zv.w;
                        }
                    }
                    auto pv = [&](int j) { return make_float2(__uint_as_float(p16[2 * j]), __uint_as_float(p16[2 * j + 1])); };
                    if (piece != rpiece) {
                        const float2 ff = make_float2(f, f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float2 v = __fmul2_rn(pv(j), __fmul2_rn(ff, make_float2(cs[2 * j], cs[2 * j + 1])));
                            if (!all_keep) {
                                const int sa = tok0 + 2 * j;
                                if (!(REV ? (zs[2 * j] <= r) : (zrr <= sa))) v.x = 0.f;
                                if (!(REV ? (zs[2 * j + 1] <= r) : (zrr <= sa + 1))) v.y = 0.f;
                            }
                            split_bf16x2(v, hi[j], lo[j]);
                        }
                    } else {
                        const float2 cc = make_float2(clr, clr);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // decay exponent: cl_r - cl_s forward, cl_s - cl_r reversed
                            const float2 cs2 = make_float2(cs[2 * j], cs[2 * j + 1]);
                            const float2 arg = REV ? __ffma2_rn(cc, make_float2(-1.f, -1.f), cs2)
                                                   : __ffma2_rn(cs2, make_float2(-1.f, -1.f), cc);
                            float2 v = __fmul2_rn(pv(j), make_float2(ex2(arg.x), ex2(arg.y)));
                            const int sa = tok0 + 2 * j;
                            if (!(REV ? (sa >= r && zs[2 * j] <= r) : (sa <= r && zrr <= sa))) v.x = 0.f;
                            if (!(REV ? (sa + 1 >= r && zs[2 * j + 1] <= r) : (sa + 1 <= r && zrr <= sa + 1))) v.y = 0.f;
                            split_bf16x2(v, hi[j], lo[j]);
                        }
                    }
                };
                auto piece_f = [&](int piece, int s0) {
                    return piece == rpiece ? 0.f : (REV ? ex2(cl[s0] - clr) : ex2(clr - cl[s0 + 31]));
                };
                auto piece_keep = [&](int s0) { return REV ? (zr[s0 + 31] <= r) : (zrr <= s0); };
                if constexpr (TC == 128) {
                    // this warp's unmasked pieces (warp-uniform)
                    static_assert(PIECES == 2, "two 32-token pieces per warp at 128-token chunks");
                    const bool lo_masked = piece_masked(2 * hf), hi_masked = piece_masked(2 * hf + 1);
                    const int npc = (lo_masked ? 0 : 1) + (hi_masked ? 0 : 1);
                    const int first = lo_masked ? 2 * hf + 1 : 2 * hf;
#pragma unroll 1
                    for (int k = 0; k < npc; ++k) {
                        const int piece = (k == 0) ? first : 2 * hf + 1;
                        const int s0 = piece * 32;
                        uint32_t pr[2][16];
                        tmem_ld16(tmem + tlane + C::C_P + (uint32_t)s0, pr[0]);
                        tmem_ld16(tmem + tlane + C::C_P + (uint32_t)(s0 + 16), pr[1]);
                        const float f = piece_f(piece, s0);
                        const bool all_keep = piece_keep(s0);
                        tmem_ld_wait();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // tokens s0 + 16h..: high parts at columns s0 + 8h.., low parts 16 further
                            uint32_t hi[8], lo[8];
                            mask16(pr[h], piece, s0 + 16 * h, f, all_keep, hi, lo);
                            tmem_st8(tmem + tlane + C::C_PB + (uint32_t)(s0 + 8 * h), hi);
                            tmem_st8(tmem + tlane + C::C_PB + (uint32_t)(s0 + 16 + 8 * h), lo);
                        }
                    }
                    tmem_st_wait();
                } else {
                    // 64-row scores: lanes 0..15 hold this warp's 16 rows; threads 0..15 take tokens
                    // s0..s0+15 of the piece, threads 16..31 tokens s0+16..s0+31 (paired-half shapes)
                    const int piece = hf;  // one 32-token piece per warp
                    if (!piece_masked(piece)) {
                        const int s0 = piece * 32;
                        uint32_t pr[16];
                        tmem_ld16x2(tmem + tlane + C::C_P + (uint32_t)s0, pr);
                        const float f = piece_f(piece, s0);
                        const bool all_keep = piece_keep(s0);
                        tmem_ld_wait();
                        uint32_t hi[8], lo[8];
                        mask16(pr, piece, s0 + 16 * (lane >> 4), f, all_keep, hi, lo);
                        // high parts of tokens s0.. at columns s0.., of s0+16.. at s0+8..; low parts 16 further
                        tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)s0, hi);
                        tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)(s0 + 16), lo);
                    } else if constexpr (C::COMPACT) {
                        // masked in place: every P product rewrites this fully masked piece
                        const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                        tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)(piece * 32), zero);
                        tmem_st8x2(tmem + tlane + C::C_PB + (uint32_t)(piece * 32 + 16), zero);
                    }
                    tmem_st_wait();
                }
            }
            tc_fence_before();
            bar_arrive(kBarPmask, kAllThreads);
            // ---- State = alpha State + dS
            wait(5);
            tc_fence_after();
            state_accumulate(alpha);
            // ---- OUT = O_intra + w_out O_inter (this warp: columns [32 hf, 32 hf + 32)), staged in the
            // 128-byte-swizzled output tile; each warp stores its own rows with a TMA store
            wait(7);
            wait(6);
            tc_fence_after();
            if (has_w) wait(3);
            {
                const int r = prow;
                const float wr = wout[r];
                uint32_t oa[OW], oi[OW];
                tmem_ld_cols<OW>(tmem + tlane + C::C_OA + hf * 32, oa);
                tmem_ld_cols<OW>(tmem + tlane + C::C_OI + hf * 32, oi);
                tmem_ld_wait();
                float o[OW];
#pragma unroll
                for (int jj = 0; jj < OW / 2; ++jj) {
                    const float2 v = __ffma2_rn(make_float2(wr, wr),
                                                make_float2(__uint_as_float(oi[2 * jj]), __uint_as_float(oi[2 * jj + 1])),
                                                make_float2(__uint_as_float(oa[2 * jj]), __uint_as_float(oa[2 * jj + 1])));
                    o[2 * jj] = v.x;
                    o[2 * jj + 1] = v.y;
                }
                {
                    const uint32_t row = sbase + C::OFF_ZS + (uint32_t)(hf * TC * 128 + prow * 128);
                    const int c0 = (ocol - hf * 32) / 4;  // this thread's first 16-byte chunk of the row
#pragma unroll
                    for (int c = 0; c < OW / 4; ++c)
                        st_shared_v4(row + (uint32_t)(((c0 + c) ^ (prow & 7)) << 4), o[c * 4], o[c * 4 + 1],
                                     o[c * 4 + 2], o[c * 4 + 3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // rows past T are clipped by the store; the Zs buffer is rewritten only after
                    // every warp's store has read its rows (the wait before the next chunk's Zs)
                    constexpr int WROWS = (TC == 128) ? 32 : 16;
                    tma_store_3d(&maps.out, zb * 64 + hf * 32, (int)t0 + q * WROWS, bh,
                                 sbase + C::OFF_ZS + (uint32_t)(hf * TC * 128 + q * WROWS * 128));
                    tma_store_commit();
                }
                if (has_w) {
                    float dot = 0.f;
                    if (t0 + prow < p.T) {
#pragma unroll
                        for (int c = 0; c < OW / 8; ++c) {
                            const uint4 qq = *reinterpret_cast<const uint4 *>(smem + C::OFF_W + sw128(r, ocol + c * 8));
                            const uint32_t words[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 fw = unpack_bf16(words[e]);
                                dot = fmaf(o[c * 8 + 2 * e], fw.x, fmaf(o[c * 8 + 2 * e + 1], fw.y, dot));
                            }
                        }
                    }
                    if (TC == 64) dot += __shfl_xor_sync(0xffffffffu, dot, 16);  // the row's other 16 columns
                    if ((TC == 128 || lane < 16) && t0 + prow < p.T) dotp[hf * TC + r] = dot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(10 + ((nc + i - v0) & 1)));  // done with this visit's decays
            // State's bf16 parts for the next chunk (this chunk's O_inter has consumed them)
            write_s_smem();
            fence_async_smem();
            tc_fence_before();
            if (has_w) {
                bar_sync(kBarMath, kMathThreads);
                if (hf == 0 && (TC == 128 || lane < 16) && t0 + prow < p.T)
                    p.wdot[((size_t)zb * p.BH + bh) * p.T + t0 + prow] = dotp[prow] + dotp[TC + prow];
            }
            bar_arrive(kBarDone, kAllThreads);
        }
        if (lane == 0) tma_store_wait_all();

        // ---- final state of the sequence
        const bool last = REV ? (seg == 0) : (seg == p.n_seg - 1);
        if (last && p.fs_mode == 1) {
#pragma unroll
            for (int c = 0; c < SW; ++c) p.fs_out[((size_t)bh * DX + srow) * p.DZ + zb * 64 + scol + c] = S[c];
        } else if (last && p.fs_mode == 2) {
            float acc = 0.f;
            if (p.fs_dot != nullptr) {
#pragma unroll
                for (int c = 0; c < SW; ++c)
                    acc = fmaf(S[c], p.fs_dot[((size_t)bh * p.DZ + zb * 64 + scol + c) * DX + srow], acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) s_red[warp] = acc;
            bar_sync(kBarMath, kMathThreads);
            if (mtid == 0) {
                float t = 0.f;
                for (int w = 0; w < 8; ++w) t += s_red[w];
                p.fs_partial[(size_t)zb * p.BH + bh] = t;
            }
        }
    }
    if (timed_out) {
        atomicOr(&p.hdr->error, kErrTimeout);
        atomicExch(&p.hdr->where, 40u + (unsigned)p.ticket_slot);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// ----------------------------------------------------------------- host side
template <int DX, int TC, bool REV>
int launch_tc_variant(const LaArgs &a, cudaStream_t s, unsigned int grid) {
    using C = TcCfg<DX, TC>;
    static std::atomic<unsigned long long> smem_set{0};  // per template instance
    const void *fn = reinterpret_cast<const void *>(la_tc_kernel<DX, TC, REV>);
    if constexpr (C::COMPACT) {
        // all of the unified L1 / shared array as shared memory, so that two blocks fit an SM
        static std::atomic<unsigned long long> carve_set{0};
        int dev = 0;
        CLA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
        const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
        if (bit == 0ull || (carve_set.load(std::memory_order_acquire) & bit) == 0ull) {
            CLA_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100),
                         "cudaFuncSetAttribute");
            carve_set.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    const int st = set_max_dynamic_smem(smem_set, fn, C::SMEM);
    if (st) return st;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    bool ok = make_map(&maps.x, a.X, DX, a.T, a.BH, TC) &&
              make_map(&maps.y, a.Y, DX, a.T, a.BH, TC) &&
              make_map(&maps.z, a.Z, a.DZ, a.T, a.BH, TC) &&
              make_map(&maps.out, a.out, a.DZ, a.T, a.BH, TC == 128 ? 32 : 16, false);
    if (ok && a.W != nullptr) ok = make_map(&maps.w, a.W, a.DZ, a.T, a.BH, TC);
    if (!ok) return fail(CLA_ERR_CUDA, "chunk_la: tensor map encoding failed");
    la_tc_kernel<DX, TC, REV><<<grid, C::NT, C::SMEM, s>>>(maps, a);
    return check_launch("la_tc_kernel");
}

int launch_tc_pass(int DX, int TC, bool REV, const LaArgs &a, cudaStream_t s, unsigned int grid) {
#define CLA_TC_CASE(dx, tc)                                                           \
    if (DX == dx && TC == tc)                                                         \
        return REV ? launch_tc_variant<dx, tc, true>(a, s, grid) : launch_tc_variant<dx, tc, false>(a, s, grid);
    CLA_TC_CASE(64, 64)
    CLA_TC_CASE(64, 128)
    CLA_TC_CASE(128, 64)
    CLA_TC_CASE(128, 128)
#undef CLA_TC_CASE
    return fail(CLA_ERR_UNSUPPORTED, "chunk_la: no tensor-core kernel for head dim %d and chunk %d", DX, TC);
}

}  // namespace
}  // namespace cla
