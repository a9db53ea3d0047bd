// chunk_la.cu -- chunkwise decayed linear attention, forward and backward,
// for GB300 (sm_103a).
//
// "Parallel Scan" (zerotofrontier.app), "The chunkwise algorithm" and "The
// backward pass of linear attention"; "Lightning Attention-2", eqs. 8, 10,
// 15, 17, 19, 20 and Algorithms 1-2 (with per-token decays in place of powers
// of one lambda).
//
// One kernel template computes every chunk product of the method.  With
// in-chunk decays D (mask), lambda (from the chunk start, including the first
// token's decay), gamma (to the chunk end, excluding the writing token's own)
// and alpha (the whole chunk), each chunk of each traversal does
//     OUT_[j] = (X_[j] Y_[j]^T . M) Z_[j] + diag(w_out) X_[j] State
//     State   = alpha State + Y_[j]^T diag(w_state) Z_[j]
// either forward in time (M = D, w_out = lambda, w_state = gamma) or reversed
// (M = D^T, w_out = gamma, w_state = lambda, chunks visited last to first):
//     forward output O:  X=Q,  Y=K,  Z=V,  State=S           (forward)
//     dQ:                X=dO, Y=V,  Z=K,  State=S^T         (forward)
//     dV:                X=K,  Y=Q,  Z=dO, State=dS          (reversed)
//     dK:                X=V,  Y=dO, Z=Q,  State=dS^T        (reversed)
// which are the four block formulas of the pages.  A block handles one
// 64-column slab of Z (and of OUT and State).
//
// Chunk parallelism ("Splitting one sequence across devices", applied across
// the blocks of one GPU): the chunks are grouped into segments; a block owns
// one segment.  Phase 1 folds the segment's chunks into one affine pair
// (alpha_seg, dState_seg) from a zero state and publishes it; decoupled
// look-back over earlier segments' pairs gives the true incoming state; the
// block publishes its outgoing state; phase 2 runs the chunk recurrence above
// from that state and writes OUT.  Phase 2 re-reads the segment's Y and Z,
// which phase 1 read shortly before (L2-resident for the segment sizes used).
//
// Two kernels implement the template.  la_tc_kernel (chunk_la_tc.cuh) runs
// every sequence with at least one full chunk: tcgen05 MMAs with the
// accumulators in tensor memory, TMA tile loads and stores, warp-specialised.
// la_chunk_kernel below runs the shorter ones (the TMA boxes are one chunk
// tall): mma.sync m16n8k16 (bf16 in, fp32 accumulate) on tiles staged in
// shared memory with cp.async (double-buffered) and XOR-swizzled rows.  Both
// keep the state in fp32 registers.  The three operands that
// are not inputs -- the masked scores, the state fed to the X State product
// and w_state * Z in the state update -- are each split into a high and a low
// bf16 part (two MMAs), so their rounding stays far below the fp32 outputs'
// tolerance; bf16 rounding of those operands alone would cost about 1% of
// the output RMS each.  Decays come from in-chunk sums of
// log a (never from long cumulative sums or ratios); a reset (log a = -inf)
// zeroes every product that spans it.
#include <cuda_bf16.h>

#include "cla_internal.cuh"
#include "mma_sync.cuh"

namespace cla {
namespace {

typedef __nv_bfloat16 bf16;

constexpr float kLog2e = 1.4426950408889634f;
// Chunks per segment (one block): the largest of kSegChoices that still
// leaves at least kMinBlocks blocks (several waves on a 152-SM part), so the
// fixed cost of a block's look-back is spread over as many chunks as the
// grid's size allows; the smallest choice otherwise.
constexpr int kSegChoices[4] = {64, 32, 16, 8};
constexpr long long kMinBlocks = 1024;
// The compact layout (d_k = d_v = chunk = 64, two blocks per SM) has short chunk visits (about
// 3k cycles), so a block's fixed cost weighs more there: it takes the rule with a quarter of the
// blocks, about one wave of two blocks per SM (measured on 4 x 16 x 8192: 4-chunk segments
// 181 / 434 us forward / backward, 8-chunk 155 / 395 us, 16-chunk 143 / 382 us, 32-chunk
// 133 / 360 us, 64-chunk (128 blocks, fewer than the SMs) 192 / 514 us).
constexpr long long kMinBlocksCompact = 256;

// ----------------------------------------------------------------- configuration
template <int DX, int TC>
struct LaCfg {
    static constexpr int NW = TC / 16;  // one warp per 16 rows of the chunk
    static constexpr int NT = NW * 32;
    static constexpr int XRB = DX * 2;  // bytes per X / Y row
    static constexpr int ZRB = 128;     // bytes per row of a 64-column Z slab
    static constexpr int S_TILES = (DX / 16) * 8 / NW;  // m16n8 state tiles per warp
    static constexpr int S_NT = S_TILES < 8 ? S_TILES : 8;
    static constexpr int S_MT = S_TILES / S_NT;
    static constexpr int X_BYTES = TC * XRB;
    static constexpr int Z_BYTES = TC * ZRB;
    static constexpr int L_BYTES = TC * 4;
    static constexpr int OFF_Y = X_BYTES;
    static constexpr int OFF_Z = 2 * X_BYTES;
    static constexpr int OFF_L = 2 * X_BYTES + Z_BYTES;
    static constexpr int STAGE = 2 * X_BYTES + Z_BYTES + L_BYTES;
    static constexpr int OFF_SB = 2 * STAGE;           // State, high bf16 part
    static constexpr int OFF_SBL = OFF_SB + DX * ZRB;  // State, low bf16 part
    static constexpr int OFF_DEC = OFF_SBL + DX * ZRB;
    static constexpr int SMEM = OFF_DEC + 4 * TC * 4 + 64;
    static_assert(S_TILES * NW == (DX / 16) * 8, "state tiles divide over warps");
    static_assert(S_NT % 2 == 0, "state n-tiles are processed in pairs");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct LaArgs {
    const bf16 *X, *Y, *Z;  // X, Y: [BH][T][DX]; Z: [BH][T][DZ]
    const float *ell;       // [BH][T] log decays
    const float *state0;    // [BH][DX][DZ] (trans0 = 0) or [BH][DZ][DX] (trans0 = 1); NULL = 0
    int trans0;
    float *out;  // [BH][T][DZ] fp32
    int fs_mode;  // final state: 0 none, 1 write fp32 [BH][DX][DZ], 2 dot with fs_dot^T
    float *fs_out;
    const float *fs_dot;  // [BH][DZ][DX]: element (row, col) of the state pairs with fs_dot[col][row]
    float *fs_partial;    // [nzb][BH]
    const bf16 *W;        // [BH][T][DZ] or NULL: per-token dot of OUT (fp32) with W
    float *wdot;          // [nzb][BH][T]
    int BH, DZ, nzb, n_chunks, seg_chunks, n_seg, ticket_slot;
    long long T;
    WsHeader *hdr;
    unsigned int *flags;  // [n_seg][BH][nzb]
    float *alpha_ws;      // [n_seg][BH][nzb]
    float4 *agg;          // [unit][S_TILES][NT] float4
    float4 *incl;
    // Incoming state of every segment, [n_seg][BH][DX][DZ] fp32 (tensor-core kernel only):
    // written after the look-back when seg_out is set; when seg_in is set, read instead of
    // running phase 1 and the look-back (seg_trans = 1: stored as [DZ][DX], i.e. the
    // transposed state of another traversal).
    float *seg_out;
    const float *seg_in;
    int seg_trans;
};

// ----------------------------------------------------------------- the kernel
template <int DX, int TC, bool REV>
__global__ void __launch_bounds__(TC * 2) la_chunk_kernel(const LaArgs p) {
    using C = LaCfg<DX, TC>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ unsigned int s_ticket, s_flag;
    __shared__ float s_alpha;
    __shared__ float s_red[C::NW];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    if (tid == 0) s_ticket = atomicAdd(&p.hdr->ticket[p.ticket_slot], 1u);
    __syncthreads();
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

    const bf16 *Xb = p.X + (size_t)bh * p.T * DX;
    const bf16 *Yb = p.Y + (size_t)bh * p.T * DX;
    const bf16 *Zb = p.Z + (size_t)bh * p.T * p.DZ + zb * 64;
    const float *Lb = p.ell + (size_t)bh * p.T;

    float *cl = reinterpret_cast<float *>(smem + C::OFF_DEC);  // in-chunk log2 sums (resets skipped)
    int *zr = reinterpret_cast<int *>(cl + TC);                // last reset index <= r, or -1
    float *wout = reinterpret_cast<float *>(zr + TC);
    float *wst = wout + TC;
    uint8_t *sb = smem + C::OFF_SB;    // State = sb + sbl (two bf16 parts), [DX][64] each
    uint8_t *sbl = smem + C::OFF_SBL;

    auto chunk_at = [&](int i) { return REV ? (c_end - 1 - i) : (c_begin + i); };

    auto load_stage = [&](int stage, int chunk, bool withX) {
        uint8_t *st = smem + stage * C::STAGE;
        const long long t0 = (long long)chunk * TC;
        constexpr int XC = C::XRB / 16;
        for (int i = tid; i < TC * XC; i += C::NT) {
            const int row = i / XC, c16 = i % XC;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            const size_t off = (size_t)(ok ? t : 0) * DX + c16 * 8;
            cp_async16(smem_u32(st + C::OFF_Y + swz<C::XRB>(row, c16)), Yb + off, ok ? 16u : 0u);
            if (withX) cp_async16(smem_u32(st + swz<C::XRB>(row, c16)), Xb + off, ok ? 16u : 0u);
        }
        for (int i = tid; i < TC * 8; i += C::NT) {
            const int row = i >> 3, c16 = i & 7;
            const long long t = t0 + row;
            const bool ok = t < p.T;
            cp_async16(smem_u32(st + C::OFF_Z + swz<C::ZRB>(row, c16)), Zb + (size_t)(ok ? t : 0) * p.DZ + c16 * 8,
                       ok ? 16u : 0u);
        }
        for (int i = tid; i < TC; i += C::NT) {
            const long long t = t0 + i;
            const bool ok = t < p.T;
            cp_async4(smem_u32(st + C::OFF_L + i * 4), Lb + (ok ? t : 0), ok ? 4u : 0u);
        }
    };

    // In-chunk decays of the chunk in `stage`; returns alpha.  Padding rows
    // past T have log a = 0 and zero data, so they change nothing.
    auto decays = [&](int stage) {
        const float *ls = reinterpret_cast<const float *>(smem + stage * C::STAGE + C::OFF_L);
        if (warp == 0) {
            constexpr int PER = TC / 32;
            float v[PER];
            int zz[PER];
            float run = 0.f;
            int lastz = -1;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int r = lane * PER + k;
                const float l = ls[r];
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
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                cl[lane * PER + k] = v[k] + ex;
                zr[lane * PER + k] = max(zz[k], zex);
            }
            __syncwarp();
            const float cL = cl[TC - 1];
            const int zL = zr[TC - 1];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int r = lane * PER + k;
                const float lam = zr[r] >= 0 ? 0.f : ex2(cl[r]);
                const float gam = zL > r ? 0.f : ex2(cL - cl[r]);
                wout[r] = REV ? gam : lam;
                wst[r] = REV ? lam : gam;
            }
            if (lane == 0) s_alpha = zL >= 0 ? 0.f : ex2(cL);
        }
        __syncthreads();
        return s_alpha;
    };

    // State fragments: warp owns S_MT x S_NT m16n8 tiles of the [DX][64] state.
    float S[C::S_MT][C::S_NT][4];
    const int tau0 = warp * C::S_TILES;
    const int mt0 = tau0 / 8, nt0 = tau0 % 8;
    auto s_row = [&](int mi, int e) { return (mt0 + mi) * 16 + g + (e >> 1) * 8; };
    auto s_col = [&](int nj, int e) { return (nt0 + nj) * 8 + tq * 2 + (e & 1); };

    // State = alpha State + Y^T diag(w_state) Z (k over the chunk's tokens).
    // The scaled B operand w_state * Z is formed in registers from the raw Z
    // fragment and split into two bf16 parts (high + low) so that its
    // rounding does not enter the state.
    auto state_update = [&](int stage, float alpha) {
        const uint8_t *ys = smem + stage * C::STAGE + C::OFF_Y;
        const uint8_t *zsrc = smem + stage * C::STAGE + C::OFF_Z;
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[mi][nj][e] *= alpha;
#pragma unroll 2
        for (int kk = 0; kk < TC / 16; ++kk) {
            // token rows of this thread's B fragment elements: 2tq, 2tq+1, 2tq+8, 2tq+9
            const float w0 = wst[kk * 16 + 2 * tq], w1 = wst[kk * 16 + 2 * tq + 1];
            const float w8 = wst[kk * 16 + 2 * tq + 8], w9 = wst[kk * 16 + 2 * tq + 9];
            uint32_t bh_[C::S_NT / 2][4], bl_[C::S_NT / 2][4];
#pragma unroll
            for (int nj = 0; nj < C::S_NT; nj += 2) {
                uint32_t b[4];
                const int brow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int bcol = nt0 + nj + (lane >> 4);
                ldsm_x4_t(smem_u32(zsrc + swz<C::ZRB>(brow, bcol)), b);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = unpack_bf16(b[q]);
                    const float x0 = f.x * ((q & 1) ? w8 : w0);
                    const float x1 = f.y * ((q & 1) ? w9 : w1);
                    const uint32_t hi = pack_bf16(x0, x1);
                    const float2 fh = unpack_bf16(hi);
                    bh_[nj / 2][q] = hi;
                    bl_[nj / 2][q] = pack_bf16(x0 - fh.x, x1 - fh.y);
                }
            }
#pragma unroll
            for (int mi = 0; mi < C::S_MT; ++mi) {
                uint32_t a[4];
                const int arow = kk * 16 + (lane & 7) + (lane >> 4) * 8;
                const int acol = (mt0 + mi) * 2 + ((lane >> 3) & 1);
                ldsm_x4_t(smem_u32(ys + swz<C::XRB>(arow, acol)), a);
#pragma unroll
                for (int nj = 0; nj < C::S_NT; nj += 2) {
                    mma16816(S[mi][nj], a, bh_[nj / 2][0], bh_[nj / 2][1]);
                    mma16816(S[mi][nj + 1], a, bh_[nj / 2][2], bh_[nj / 2][3]);
                    mma16816(S[mi][nj], a, bl_[nj / 2][0], bl_[nj / 2][1]);
                    mma16816(S[mi][nj + 1], a, bl_[nj / 2][2], bl_[nj / 2][3]);
                }
            }
        }
    };

    // State as two bf16 parts (high + low) for the X State product.
    auto write_sb = [&]() {
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = s_row(mi, h * 2), col = s_col(nj, 0);
                    const uint32_t off = swz<C::ZRB>(row, col >> 3) + (col & 7) * 2;
                    const float x0 = S[mi][nj][h * 2], x1 = S[mi][nj][h * 2 + 1];
                    const uint32_t hi = pack_bf16(x0, x1);
                    const float2 fh = unpack_bf16(hi);
                    *reinterpret_cast<uint32_t *>(sb + off) = hi;
                    *reinterpret_cast<uint32_t *>(sbl + off) = pack_bf16(x0 - fh.x, x1 - fh.y);
                }
    };

    auto ws_index = [&](int i) { return unit * (size_t)(C::S_TILES * C::NT) + (size_t)i * C::NT + tid; };

    // ------------------------------------------------ phase 1: segment aggregate
#pragma unroll
    for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
        for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[mi][nj][e] = 0.f;
    float alpha_seg = 1.f;
    load_stage(0, chunk_at(0), false);
    cp_async_commit();
    if (nc > 1) load_stage(1, chunk_at(1), false);
    cp_async_commit();
    for (int i = 0; i < nc; ++i) {
        const int stage = i & 1;
        cp_async_wait<1>();
        __syncthreads();
        const float alpha = decays(stage);
        alpha_seg *= alpha;
        __syncthreads();
        state_update(stage, alpha);
        __syncthreads();
        if (i + 2 < nc) load_stage(stage, chunk_at(i + 2), false);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ------------------------------------------------ look-back for the incoming state
    const bool first = REV ? (seg == p.n_seg - 1) : (seg == 0);
    float Sin[C::S_MT][C::S_NT][4];
    auto load_state0 = [&](float (&dst)[C::S_MT][C::S_NT][4], float scale, bool add) {
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = 0.f;
                    if (p.state0 != nullptr) {
                        const int row = s_row(mi, e), col = zb * 64 + s_col(nj, e);
                        v = p.trans0 ? p.state0[((size_t)bh * p.DZ + col) * DX + row]
                                     : p.state0[((size_t)bh * DX + row) * p.DZ + col];
                    }
                    dst[mi][nj][e] = add ? fmaf(scale, v, dst[mi][nj][e]) : v;
                }
    };
    if (first) {
        load_state0(Sin, 1.f, false);
    } else {
        // publish this segment's aggregate
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
                __stcg(p.agg + ws_index(mi * C::S_NT + nj),
                       make_float4(S[mi][nj][0], S[mi][nj][1], S[mi][nj][2], S[mi][nj][3]));
        if (tid == 0) p.alpha_ws[unit] = alpha_seg;
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(p.flags + unit, 1u);
        // walk back (forward traversal: toward seg 0; reversed: toward the end)
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e) Sin[mi][nj][e] = 0.f;
        float accA = 1.f;
        int j = REV ? seg + 1 : seg - 1;
        while (true) {
            const size_t up = ((size_t)j * p.BH + bh) * p.nzb + zb;
            if (tid == 0) {
                const unsigned int f = wait_flag(p.flags + up, p.hdr, 10u + (unsigned)p.ticket_slot);
                s_flag = f;
                if (f == 1u) s_alpha = ld_cg(p.alpha_ws + up);
            }
            __syncthreads();
            const unsigned int f = s_flag;
            const float pa = s_alpha;
            __syncthreads();
            if (f == 2u) {
#pragma unroll
                for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
                    for (int nj = 0; nj < C::S_NT; ++nj) {
                        const float4 v = ld_cg4(p.incl + up * (size_t)(C::S_TILES * C::NT) +
                                                (size_t)(mi * C::S_NT + nj) * C::NT + tid);
                        Sin[mi][nj][0] = fmaf(accA, v.x, Sin[mi][nj][0]);
                        Sin[mi][nj][1] = fmaf(accA, v.y, Sin[mi][nj][1]);
                        Sin[mi][nj][2] = fmaf(accA, v.z, Sin[mi][nj][2]);
                        Sin[mi][nj][3] = fmaf(accA, v.w, Sin[mi][nj][3]);
                    }
                break;
            } else if (f == 1u) {
#pragma unroll
                for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
                    for (int nj = 0; nj < C::S_NT; ++nj) {
                        const float4 v = ld_cg4(p.agg + up * (size_t)(C::S_TILES * C::NT) +
                                                (size_t)(mi * C::S_NT + nj) * C::NT + tid);
                        Sin[mi][nj][0] = fmaf(accA, v.x, Sin[mi][nj][0]);
                        Sin[mi][nj][1] = fmaf(accA, v.y, Sin[mi][nj][1]);
                        Sin[mi][nj][2] = fmaf(accA, v.z, Sin[mi][nj][2]);
                        Sin[mi][nj][3] = fmaf(accA, v.w, Sin[mi][nj][3]);
                    }
                accA *= pa;
                j = REV ? j + 1 : j - 1;
                if (j < 0 || j >= p.n_seg) {  // reached the sequence's edge: the initial state
                    load_state0(Sin, accA, true);
                    break;
                }
            } else {
                break;  // a wait gave up; reported through the workspace
            }
        }
    }
    // publish the outgoing state: alpha_seg * Sin + aggregate
#pragma unroll
    for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
        for (int nj = 0; nj < C::S_NT; ++nj)
            __stcg(p.incl + ws_index(mi * C::S_NT + nj),
                   make_float4(fmaf(alpha_seg, Sin[mi][nj][0], S[mi][nj][0]),
                               fmaf(alpha_seg, Sin[mi][nj][1], S[mi][nj][1]),
                               fmaf(alpha_seg, Sin[mi][nj][2], S[mi][nj][2]),
                               fmaf(alpha_seg, Sin[mi][nj][3], S[mi][nj][3])));
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release(p.flags + unit, 2u);

    // ------------------------------------------------ phase 2: outputs
#pragma unroll
    for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
        for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[mi][nj][e] = Sin[mi][nj][e];
    write_sb();
    load_stage(0, chunk_at(0), true);
    cp_async_commit();
    if (nc > 1) load_stage(1, chunk_at(1), true);
    cp_async_commit();
    const int r0 = warp * 16;
    for (int i = 0; i < nc; ++i) {
        const int stage = i & 1;
        const int chunk = chunk_at(i);
        uint8_t *st = smem + stage * C::STAGE;
        cp_async_wait<1>();
        __syncthreads();
        const float alpha = decays(stage);
        // ---- OUT rows r0..r0+15 = w_out * (X State) + (X Y^T . M) Z
        float o[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DX / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(smem_u32(st + swz<C::XRB>(r0 + (lane & 7) + ((lane >> 3) & 1) * 8, kk * 2 + (lane >> 4))), a);
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) {
                uint32_t b[4], bl[4];
                const uint32_t off = swz<C::ZRB>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, nj * 2 + (lane >> 4));
                ldsm_x4_t(smem_u32(sb + off), b);
                ldsm_x4_t(smem_u32(sbl + off), bl);
                mma16816(o[2 * nj], a, b[0], b[1]);
                mma16816(o[2 * nj + 1], a, b[2], b[3]);
                mma16816(o[2 * nj], a, bl[0], bl[1]);
                mma16816(o[2 * nj + 1], a, bl[2], bl[3]);
            }
        }
        {
            const float w0 = wout[r0 + g], w1 = wout[r0 + g + 8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o[j][0] *= w0;
                o[j][1] *= w0;
                o[j][2] *= w1;
                o[j][3] *= w1;
            }
        }
#pragma unroll
        for (int cb = 0; cb < TC / 64; ++cb) {
            if (!REV && 64 * cb > r0 + 15) continue;  // entirely above the diagonal
            if (REV && 64 * cb + 63 < r0) continue;   // entirely below
            float pc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) pc[j][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DX / 16; ++kk) {
                uint32_t a[4];
                ldsm_x4(smem_u32(st + swz<C::XRB>(r0 + (lane & 7) + ((lane >> 3) & 1) * 8, kk * 2 + (lane >> 4))), a);
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    const int n0 = 64 * cb + 16 * nj;
                    if (!REV && n0 > r0 + 15) continue;
                    if (REV && n0 + 15 < r0) continue;
                    uint32_t b[4];
                    ldsm_x4(smem_u32(st + C::OFF_Y +
                                     swz<C::XRB>(n0 + (lane & 7) + (lane >> 4) * 8, kk * 2 + ((lane >> 3) & 1))),
                            b);
                    mma16816(pc[2 * nj], a, b[0], b[1]);
                    mma16816(pc[2 * nj + 1], a, b[2], b[3]);
                }
            }
            // mask and in-chunk decay
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = r0 + g + (e >> 1) * 8;
                    const int s = 64 * cb + 8 * j + 2 * tq + (e & 1);
                    float m;
                    if (!REV) m = (s <= r && zr[r] <= s) ? ex2(cl[r] - cl[s]) : 0.f;
                    else m = (s >= r && zr[s] <= r) ? ex2(cl[s] - cl[r]) : 0.f;
                    pc[j][e] *= m;
                }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int s0 = 64 * cb + 16 * kk;
                if (!REV && s0 > r0 + 15) continue;
                if (REV && s0 + 15 < r0) continue;
                // masked scores as two bf16 parts (high + low)
                uint32_t a[4], al[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float x0 = pc[2 * kk + (q >> 1)][(q & 1) * 2];
                    const float x1 = pc[2 * kk + (q >> 1)][(q & 1) * 2 + 1];
                    a[q] = pack_bf16(x0, x1);
                    const float2 fh = unpack_bf16(a[q]);
                    al[q] = pack_bf16(x0 - fh.x, x1 - fh.y);
                }
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    uint32_t b[4];
                    ldsm_x4_t(smem_u32(st + C::OFF_Z +
                                       swz<C::ZRB>(s0 + (lane & 7) + ((lane >> 3) & 1) * 8, nj * 2 + (lane >> 4))),
                              b);
                    mma16816(o[2 * nj], a, b[0], b[1]);
                    mma16816(o[2 * nj + 1], a, b[2], b[3]);
                    mma16816(o[2 * nj], al, b[0], b[1]);
                    mma16816(o[2 * nj + 1], al, b[2], b[3]);
                }
            }
        }
        const long long t0 = (long long)chunk * TC;
        // ---- optional per-token dot of OUT with W (fp32, before rounding)
        if (p.W != nullptr) {
            float d0 = 0.f, d1 = 0.f;
            const long long ta = t0 + r0 + g, tb = ta + 8;
            const bf16 *Wb = p.W + (size_t)bh * p.T * p.DZ + zb * 64;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = 8 * j + 2 * tq;
                if (ta < p.T) {
                    const float2 w = unpack_bf16(__ldg(reinterpret_cast<const unsigned int *>(Wb + (size_t)ta * p.DZ + col)));
                    d0 = fmaf(o[j][0], w.x, fmaf(o[j][1], w.y, d0));
                }
                if (tb < p.T) {
                    const float2 w = unpack_bf16(__ldg(reinterpret_cast<const unsigned int *>(Wb + (size_t)tb * p.DZ + col)));
                    d1 = fmaf(o[j][2], w.x, fmaf(o[j][3], w.y, d1));
                }
            }
            d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
            d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
            d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
            if (tq == 0) {
                float *wd = p.wdot + ((size_t)zb * p.BH + bh) * p.T;
                if (ta < p.T) wd[ta] = d0;
                if (tb < p.T) wd[tb] = d1;
            }
        }
        // ---- OUT (fp32): each quad of lanes writes 32 contiguous bytes of a row
        {
            float *Ob = p.out + (size_t)bh * p.T * p.DZ + zb * 64;
            const long long ta = t0 + r0 + g, tb = ta + 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = 8 * j + 2 * tq;
                if (ta < p.T) __stcs(reinterpret_cast<float2 *>(Ob + (size_t)ta * p.DZ + col), make_float2(o[j][0], o[j][1]));
                if (tb < p.T) __stcs(reinterpret_cast<float2 *>(Ob + (size_t)tb * p.DZ + col), make_float2(o[j][2], o[j][3]));
            }
        }
        __syncthreads();  // every warp done with the State copy
        state_update(stage, alpha);
        write_sb();
        __syncthreads();
        if (i + 2 < nc) load_stage(stage, chunk_at(i + 2), true);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ------------------------------------------------ final state of the sequence
    const bool last = REV ? (seg == 0) : (seg == p.n_seg - 1);
    if (last && p.fs_mode == 1) {
#pragma unroll
        for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
            for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    p.fs_out[((size_t)bh * DX + s_row(mi, e)) * p.DZ + zb * 64 + s_col(nj, e)] = S[mi][nj][e];
    } else if (last && p.fs_mode == 2) {
        float acc = 0.f;
        if (p.fs_dot != nullptr) {
#pragma unroll
            for (int mi = 0; mi < C::S_MT; ++mi)
#pragma unroll
                for (int nj = 0; nj < C::S_NT; ++nj)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc = fmaf(S[mi][nj][e],
                                   p.fs_dot[((size_t)bh * p.DZ + zb * 64 + s_col(nj, e)) * DX + s_row(mi, e)], acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_red[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < C::NW; ++w) t += s_red[w];
            p.fs_partial[(size_t)zb * p.BH + bh] = t;
        }
    }
}

// dlog_a_u = sum_{t >= u} (sum_zb qdq - sum_zb kdk)_t + sum_zb <dS_T, S_T> partials,
// as a reverse scan over tiles of kFinTile tokens: la_dlog_tile_sums_kernel
// reduces each tile, la_dlog_finalize_kernel scans a tile and adds the sum of
// every later tile and the final-state term.  Both grids are tiles x B*H
// blocks, block = bh * tiles + tile;
// every sum runs in a fixed order, so results do not depend on scheduling.
constexpr int kFinThreads = 256;
constexpr int kFinPer = 8;  // consecutive tokens per thread in the scan
constexpr int kFinTile = kFinThreads * kFinPer;

__device__ __forceinline__ float dlog_delta(const float *__restrict__ qdq, const float *__restrict__ kdk, int nzb,
                                            int BH, int bh, long long T, long long t) {
    float d = 0.f;
    for (int z = 0; z < nzb; ++z) {
        d += qdq[((size_t)z * BH + bh) * T + t];
        d -= kdk[((size_t)z * BH + bh) * T + t];
    }
    return d;
}

__global__ void __launch_bounds__(kFinThreads) la_dlog_tile_sums_kernel(const float *__restrict__ qdq,
                                                                        const float *__restrict__ kdk,
                                                                        float *__restrict__ tsum, int nzb, int BH,
                                                                        long long T, int n_tiles) {
    __shared__ float s_w[kFinThreads / 32];
    const int tile = (int)(blockIdx.x % (unsigned)n_tiles), bh = (int)(blockIdx.x / (unsigned)n_tiles);
    const int tid = threadIdx.x;
    const long long t0 = (long long)tile * kFinTile;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kFinPer; ++k) {
        const long long t = t0 + k * kFinThreads + tid;
        if (t < T) acc += dlog_delta(qdq, kdk, nzb, BH, bh, T, t);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((tid & 31) == 0) s_w[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < kFinThreads / 32; ++w) t += s_w[w];
        tsum[(size_t)bh * n_tiles + tile] = t;
    }
}

__global__ void __launch_bounds__(kFinThreads) la_dlog_finalize_kernel(
    const float *__restrict__ qdq, const float *__restrict__ kdk, const float *__restrict__ fsp,
    const float *__restrict__ tsum, float *__restrict__ dlog, int nzb, int BH, long long T, int n_tiles) {
    // tile staged with one pad word per 8, so both the coalesced pass (consecutive
    // threads, consecutive tokens) and the per-thread pass (8 consecutive tokens) are conflict-free
    __shared__ float sh[kFinTile + kFinTile / kFinPer];
    __shared__ float s_w[kFinThreads / 32];
    __shared__ float s_off;
    const int tile = (int)(blockIdx.x % (unsigned)n_tiles), bh = (int)(blockIdx.x / (unsigned)n_tiles);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long t0 = (long long)tile * kFinTile;
#pragma unroll
    for (int k = 0; k < kFinPer; ++k) {
        const int e = k * kFinThreads + tid;
        const long long t = t0 + e;
        sh[e + e / kFinPer] = (t < T) ? dlog_delta(qdq, kdk, nzb, BH, bh, T, t) : 0.f;
    }
    if (warp == 0) {  // offset of this tile: every later tile plus the final-state term
        float o = 0.f;
        for (int j = tile + 1 + lane; j < n_tiles; j += 32) o += tsum[(size_t)bh * n_tiles + j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) o += __shfl_xor_sync(0xffffffffu, o, off);
        if (lane == 0) {
            float tail = 0.f;
            for (int z = 0; z < nzb; ++z) tail += fsp[(size_t)z * BH + bh];
            s_off = o + tail;
        }
    }
    __syncthreads();
    float v[kFinPer];
    float run = 0.f;
#pragma unroll
    for (int j = kFinPer - 1; j >= 0; --j) {
        run += sh[tid * (kFinPer + 1) + j];
        v[j] = run;
    }
    // exclusive suffix sum of the thread totals (threads after this one)
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += o;
    }
    if (lane == 0) s_w[warp] = incl;
    __syncthreads();
    float after = s_off + (incl - run);
    for (int w = warp + 1; w < kFinThreads / 32; ++w) after += s_w[w];
#pragma unroll
    for (int j = 0; j < kFinPer; ++j) sh[tid * (kFinPer + 1) + j] = v[j] + after;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kFinPer; ++k) {
        const int e = k * kFinThreads + tid;
        const long long t = t0 + e;
        if (t < T) dlog[(size_t)bh * T + t] = sh[e + e / kFinPer];
    }
}

// ----------------------------------------------------------------- host side
struct LaPlan {
    int TC, DXmax, n_chunks, seg_chunks, n_seg, nzb_max;
    size_t units;
    size_t off_flags, off_alpha, off_agg, off_incl, off_qdq, off_kdk, off_fsp, off_tsum, off_seg, total;
    int fin_tiles;
};

LaPlan la_plan(int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int chunk) {
    LaPlan p;
    p.TC = chunk;
    p.DXmax = (int)(dk > dv ? dk : dv);
    p.n_chunks = (int)((T + chunk - 1) / chunk);
    p.nzb_max = (int)((dk > dv ? dk : dv) / 64);
    const size_t BH = (size_t)B * H;
    p.seg_chunks = kSegChoices[3];
    const long long min_blocks = (dk == 64 && dv == 64 && chunk == 64) ? kMinBlocksCompact : kMinBlocks;
    for (int c : kSegChoices) {
        const long long nseg = (p.n_chunks + c - 1) / c;
        if (nseg * (long long)BH * p.nzb_max >= min_blocks) {
            p.seg_chunks = c;
            break;
        }
    }
    p.n_seg = (p.n_chunks + p.seg_chunks - 1) / p.seg_chunks;
    if (p.n_seg < 1) p.n_seg = 1;
    p.units = (size_t)p.n_seg * BH * p.nzb_max;
    const size_t state_floats = (size_t)p.DXmax * 64;
    p.off_flags = sizeof(WsHeader);
    p.off_alpha = align_up(p.off_flags + p.units * 4, 256);
    p.off_agg = align_up(p.off_alpha + p.units * 4, 256);
    p.off_incl = align_up(p.off_agg + p.units * state_floats * 4, 256);
    p.off_qdq = align_up(p.off_incl + p.units * state_floats * 4, 256);
    p.off_kdk = align_up(p.off_qdq + (size_t)p.nzb_max * BH * T * 4, 256);
    p.off_fsp = align_up(p.off_kdk + (size_t)p.nzb_max * BH * T * 4, 256);
    p.off_tsum = align_up(p.off_fsp + (size_t)p.nzb_max * BH * 4, 256);
    p.fin_tiles = (int)((T + kFinTile - 1) / kFinTile);
    if (p.fin_tiles < 1) p.fin_tiles = 1;
    // the backward's adjoint state entering each segment, written by the dV traversal and
    // read (transposed) by the dK traversal: [n_seg][BH][dk][dv] fp32
    p.off_seg = align_up(p.off_tsum + (size_t)p.fin_tiles * BH * 4, 256);
    p.total = align_up(p.off_seg + (size_t)p.n_seg * BH * (size_t)dk * (size_t)dv * 4, 256);
    return p;
}

template <int DX, int TC, bool REV>
int launch_variant(const LaArgs &a, cudaStream_t s, unsigned int grid) {
    using C = LaCfg<DX, TC>;
    static std::atomic<unsigned long long> smem_set{0};  // per template instance
    const int st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(la_chunk_kernel<DX, TC, REV>), C::SMEM);
    if (st) return st;
    la_chunk_kernel<DX, TC, REV><<<grid, C::NT, C::SMEM, s>>>(a);
    return check_launch("la_chunk_kernel");
}

int launch_pass(int DX, int TC, bool REV, const LaArgs &a, cudaStream_t s, unsigned int grid) {
#define CLA_LA_CASE(dx, tc)                                                     \
    if (DX == dx && TC == tc)                                                   \
        return REV ? launch_variant<dx, tc, true>(a, s, grid) : launch_variant<dx, tc, false>(a, s, grid);
    CLA_LA_CASE(64, 64)
    CLA_LA_CASE(64, 128)
    CLA_LA_CASE(128, 64)
    CLA_LA_CASE(128, 128)
#undef CLA_LA_CASE
    return fail(CLA_ERR_UNSUPPORTED, "chunk_la: no kernel for head dim %d and chunk %d", DX, TC);
}

// Non-negative sizes the kernels and the plan handle: B*H <= 2^24, T < 2^31 (the
// tensor-map loads take 32-bit token coordinates; one head that long would not
// fit device memory anyway), B*H*T <= 2^40 (so no workspace offset can overflow) and every grid, at
// most one block per chunk and 64 columns of 128, below 2^31 blocks.
bool la_sizes_fit(int64_t B, int64_t H, int64_t T, int chunk) {
    if (!product_below({B, H}, 16777217.0) || T > kMaxTokens) return false;
    if (!product_below({B, H, T}, 1099511627777.0)) return false;
    const int64_t n_chunks = (T + chunk - 1) / chunk, fin_tiles = (T + kFinTile - 1) / kFinTile;
    return product_below({B, H, n_chunks, 2}, 2147483648.0) && product_below({B, H, fin_tiles}, 2147483648.0);
}

int la_validate(const char *fn, int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int chunk) {
    if (B < 0 || H < 0 || T < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!((dk == 64 || dk == 128) && (dv == 64 || dv == 128)))
        return fail(CLA_ERR_UNSUPPORTED, "%s: head dims must be 64 or 128 (got %lld, %lld)", fn, (long long)dk,
                    (long long)dv);
    if (chunk != 64 && chunk != 128) return fail(CLA_ERR_UNSUPPORTED, "%s: chunk must be 64 or 128", fn);
    if (!la_sizes_fit(B, H, T, chunk)) return fail(CLA_ERR_UNSUPPORTED, "%s: size out of range for one launch", fn);
    return CLA_OK;
}

LaArgs base_args(const LaPlan &pl, void *ws, int64_t BH, int64_t T) {
    LaArgs a;
    memset(&a, 0, sizeof(a));
    char *w = static_cast<char *>(ws);
    a.hdr = reinterpret_cast<WsHeader *>(w);
    a.flags = reinterpret_cast<unsigned int *>(w + pl.off_flags);
    a.alpha_ws = reinterpret_cast<float *>(w + pl.off_alpha);
    a.agg = reinterpret_cast<float4 *>(w + pl.off_agg);
    a.incl = reinterpret_cast<float4 *>(w + pl.off_incl);
    a.BH = (int)BH;
    a.T = T;
    a.n_chunks = pl.n_chunks;
    a.seg_chunks = pl.seg_chunks;
    a.n_seg = pl.n_seg;
    return a;
}

}  // namespace
}  // namespace cla

#include "chunk_la_tc.cuh"

namespace cla {
namespace {
// The tensor-core kernel needs at least one full chunk per head (its tile
// boxes are one chunk tall); shorter sequences use the mma.sync kernel.
int run_pass(int DX, int TC, bool REV, const LaArgs &a, cudaStream_t s, unsigned int grid) {
    if (a.T >= TC && tensor_map_encoder() != nullptr) return launch_tc_pass(DX, TC, REV, a, s, grid);
    return launch_pass(DX, TC, REV, a, s, grid);
}
}  // namespace
}  // namespace cla

using namespace cla;

// Sizes, head dims and chunk that the fwd / bwd calls accept (la_validate without its message).
static bool la_supported(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk) {
    return B >= 0 && H >= 0 && T >= 0 && (dim_k == 64 || dim_k == 128) && (dim_v == 64 || dim_v == 128) &&
           (chunk == 64 || chunk == 128) && la_sizes_fit(B, H, T, chunk);
}

extern "C" size_t cla_chunk_la_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                              int chunk) {
    if (!la_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    return la_plan(B, H, T, dim_k, dim_v, chunk).total;
}

extern "C" size_t cla_chunk_la_workspace(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk) {
    return cla_chunk_la_workspace_size(B, H, T, dim_k, dim_v, chunk);
}

extern "C" size_t cla_chunk_la_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                                         int chunk) {
    if (!la_supported(B, H, T, dim_k, dim_v, chunk)) return 0;
    const LaPlan pl = la_plan(B, H, T, dim_k, dim_v, chunk);
    return (size_t)pl.n_seg * (size_t)(B * H) * (size_t)dim_k * (size_t)dim_v * sizeof(float);
}

namespace {
int chunk_la_fwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *log_decay, const float *S0, float *o, float *ST, float *ckpt, int64_t B,
                      int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                      void *stream) {
    clear_error();
    int st = la_validate(fn, B, H, T, dim_k, dim_v, chunk);
    if (st) return st;
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
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, o must be 16-byte aligned", fn);
    // the state is read in 16-byte rows
    if (S0 && !aligned16(S0)) return fail(CLA_ERR_INVALID_ARG, "%s: S0 must be 16-byte aligned", fn);
    if (!aligned_or_null({log_decay, ST}, 4)) return fail(CLA_ERR_INVALID_ARG, "%s: log_decay, ST misaligned", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    if (ckpt && !aligned16(ckpt)) return fail(CLA_ERR_INVALID_ARG, "%s: ckpt must be 16-byte aligned", fn);
    const LaPlan pl = la_plan(B, H, T, dim_k, dim_v, chunk);
    if (ws_bytes < pl.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, pl.total);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_agg, s), fn);
    LaArgs a = base_args(pl, ws, BH, T);
    a.X = reinterpret_cast<const bf16 *>(q);
    a.Y = reinterpret_cast<const bf16 *>(k);
    a.Z = reinterpret_cast<const bf16 *>(v);
    a.ell = log_decay;
    a.state0 = S0;
    a.trans0 = 0;
    a.out = o;
    a.fs_mode = ST ? 1 : 0;
    a.fs_out = ST;
    a.DZ = (int)dim_v;
    a.nzb = (int)(dim_v / 64);
    a.ticket_slot = 0;
    a.seg_out = ckpt;  // [n_seg][BH][dim_k][dim_v]: the state entering each segment
    const unsigned int grid = (unsigned int)((size_t)pl.n_seg * BH * a.nzb);
    return run_pass((int)dim_k, chunk, false, a, s, grid);
}

int chunk_la_bwd_impl(const char *fn, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *log_decay, const float *S0, const uint16_t *dO, const float *dST, float *dq,
                      float *dk, float *dv, float *dlog_decay, float *dS0, const float *ckpt, int64_t B, int64_t H,
                      int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                      void *stream) {
    clear_error();
    int st = la_validate(fn, B, H, T, dim_k, dim_v, chunk);
    if (st) return st;
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
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return fail(CLA_ERR_INVALID_ARG, "%s: q, k, v, dO, dq, dk, dv must be 16-byte aligned", fn);
    // dST starts the reverse traversal and is read in 16-byte rows
    if (dST && !aligned16(dST)) return fail(CLA_ERR_INVALID_ARG, "%s: dST must be 16-byte aligned", fn);
    if (!aligned_or_null({log_decay, S0, dlog_decay, dS0}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: log_decay, S0, dlog_decay, dS0 misaligned", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    if (ckpt && !aligned16(ckpt)) return fail(CLA_ERR_INVALID_ARG, "%s: ckpt must be 16-byte aligned", fn);
    const LaPlan pl = la_plan(B, H, T, dim_k, dim_v, chunk);
    if (ws_bytes < pl.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, pl.total);
    char *w = static_cast<char *>(ws);
    float *qdq = reinterpret_cast<float *>(w + pl.off_qdq);
    float *kdk = reinterpret_cast<float *>(w + pl.off_kdk);
    float *fsp = reinterpret_cast<float *>(w + pl.off_fsp);

    // pass 1 (forward order): dQ = [(dO V^T) . D] K + diag(lambda) dO S^T, rebuilding S
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_agg, s), fn);
    LaArgs a = base_args(pl, ws, BH, T);
    a.X = reinterpret_cast<const bf16 *>(dO);
    a.Y = reinterpret_cast<const bf16 *>(v);
    a.Z = reinterpret_cast<const bf16 *>(k);
    a.ell = log_decay;
    a.state0 = S0;
    a.trans0 = 1;
    a.out = dq;
    a.fs_mode = 2;
    a.fs_dot = dST;
    a.fs_partial = fsp;
    a.W = reinterpret_cast<const bf16 *>(q);
    a.wdot = qdq;
    a.DZ = (int)dim_k;
    a.nzb = (int)(dim_k / 64);
    a.ticket_slot = 0;
    // its state is the transpose of the forward's: with the forward's checkpoint each segment
    // starts from the saved state (no phase 1, no look-back)
    a.seg_in = ckpt;
    a.seg_trans = 1;
    unsigned int grid = (unsigned int)((size_t)pl.n_seg * BH * a.nzb);
    st = run_pass((int)dim_v, chunk, false, a, s, grid);
    if (st) return st;

    // pass 2 (reverse order): dV = [(Q K^T) . D]^T dO + diag(gamma) K dS, carrying dS
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_agg, s), fn);
    a = base_args(pl, ws, BH, T);
    a.X = reinterpret_cast<const bf16 *>(k);
    a.Y = reinterpret_cast<const bf16 *>(q);
    a.Z = reinterpret_cast<const bf16 *>(dO);
    a.ell = log_decay;
    a.state0 = dST;
    a.trans0 = 0;
    a.out = dv;
    a.fs_mode = dS0 ? 1 : 0;
    a.fs_out = dS0;
    a.DZ = (int)dim_v;
    a.nzb = (int)(dim_v / 64);
    a.ticket_slot = 1;
    a.seg_out = reinterpret_cast<float *>(w + pl.off_seg);
    grid = (unsigned int)((size_t)pl.n_seg * BH * a.nzb);
    st = run_pass((int)dim_k, chunk, true, a, s, grid);
    if (st) return st;

    // pass 3 (reverse order): dK = [(dO V^T) . D]^T Q + diag(gamma) V dS^T, with dS^T
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, pl.off_agg, s), fn);
    a = base_args(pl, ws, BH, T);
    a.X = reinterpret_cast<const bf16 *>(v);
    a.Y = reinterpret_cast<const bf16 *>(dO);
    a.Z = reinterpret_cast<const bf16 *>(q);
    a.ell = log_decay;
    a.state0 = dST;
    a.trans0 = 1;
    a.out = dk;
    a.W = reinterpret_cast<const bf16 *>(k);
    a.wdot = kdk;
    a.DZ = (int)dim_k;
    a.nzb = (int)(dim_k / 64);
    a.ticket_slot = 2;
    // its adjoint state is the transpose of pass 2's: each segment starts from the state pass 2
    // saved (the tensor-core kernel skips its phase 1 and look-back; the mma.sync kernel, used
    // when T is shorter than a chunk, recomputes it)
    a.seg_in = reinterpret_cast<const float *>(w + pl.off_seg);
    a.seg_trans = 1;
    grid = (unsigned int)((size_t)pl.n_seg * BH * a.nzb);
    st = run_pass((int)dim_v, chunk, true, a, s, grid);
    if (st) return st;

    // decay gradient: suffix sums of q.dq - k.dk plus <dS_T, S_T>
    if (dlog_decay) {
        float *tsum = reinterpret_cast<float *>(w + pl.off_tsum);
        const unsigned int fgrid = (unsigned int)((size_t)pl.fin_tiles * BH);
        la_dlog_tile_sums_kernel<<<fgrid, kFinThreads, 0, s>>>(qdq, kdk, tsum, (int)(dim_k / 64), (int)BH, T,
                                                               pl.fin_tiles);
        st = check_launch("la_dlog_tile_sums_kernel");
        if (st) return st;
        la_dlog_finalize_kernel<<<fgrid, kFinThreads, 0, s>>>(qdq, kdk, fsp, tsum, dlog_decay, (int)(dim_k / 64),
                                                              (int)BH, T, pl.fin_tiles);
        st = check_launch("la_dlog_finalize_kernel");
    }
    return st;
}
}  // namespace

extern "C" int cla_chunk_la_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                const float *S0, float *o, float *ST, int64_t B, int64_t H, int64_t T,
                                int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    return chunk_la_fwd_impl("cla_chunk_la_fwd", q, k, v, log_decay, S0, o, ST, nullptr, B, H, T, dim_k, dim_v,
                             chunk, ws, ws_bytes, stream);
}

extern "C" int cla_chunk_la_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const float *log_decay, const float *S0, float *o, float *ST, float *ckpt,
                                     int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk,
                                     void *ws, size_t ws_bytes, void *stream) {
    return chunk_la_fwd_impl("cla_chunk_la_fwd_ckpt", q, k, v, log_decay, S0, o, ST, ckpt, B, H, T, dim_k, dim_v,
                             chunk, ws, ws_bytes, stream);
}

extern "C" int cla_chunk_la_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *log_decay,
                                const float *S0, const uint16_t *dO, const float *dST, float *dq, float *dk,
                                float *dv, float *dlog_decay, float *dS0, int64_t B, int64_t H, int64_t T,
                                int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    return chunk_la_bwd_impl("cla_chunk_la_bwd", q, k, v, log_decay, S0, dO, dST, dq, dk, dv, dlog_decay, dS0,
                             nullptr, B, H, T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}

extern "C" int cla_chunk_la_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     const float *log_decay, const float *S0, const uint16_t *dO,
                                     const float *dST, float *dq, float *dk, float *dv, float *dlog_decay,
                                     float *dS0, const float *ckpt, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                                     int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream) {
    return chunk_la_bwd_impl("cla_chunk_la_bwd_ckpt", q, k, v, log_decay, S0, dO, dST, dq, dk, dv, dlog_decay,
                             dS0, ckpt, B, H, T, dim_k, dim_v, chunk, ws, ws_bytes, stream);
}
