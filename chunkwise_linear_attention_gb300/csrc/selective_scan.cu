// selective_scan.cu -- selective (Mamba-1 style) diagonal scan, forward and
// backward, for GB300 (sm_103a).
//
// "Parallel Scan" (zerotofrontier.app), "Scans over vector and matrix states"
// (a diagonal transition per channel), "When a scan is the wrong tool"
// (Mamba's kernel: discretise on chip, keep the (B, T, D, N) state out of HBM,
// recompute states in the backward pass) and "The backward pass is a scan in
// reverse".
//
// Per channel d and state entry n: a = exp(delta A), b = delta B_t[n] x,
// h_t = a h_{t-1} + b, y_t = sum_n C_t[n] h_t.  The decays and inputs are
// formed in registers and never stored.
//
// Forward: one thread per channel holds all N = 16 state entries; a block owns
// 128 channels x one 64-step chunk.  Phase 1 folds the chunk into one affine
// pair per (channel, n) -- the product of the decays is exp(A sum delta), the
// composed input is accumulated step by step -- and publishes it; decoupled
// look-back over earlier chunks gives the state entering the chunk, which is
// also saved as the backward's checkpoint; phase 2 re-runs the chunk and
// writes y.
//
// Backward: two threads per channel (8 state entries each), blocks visit the
// chunks last to first.  Pass A recomputes the chunk's states from the
// checkpoint (keeping the state at every 8th step in shared memory) and folds
// the adjoint recurrence hbar_t = C_t[n] dy_t + a_{t+1} hbar_{t+1} over the
// chunk into one pair; look-back over later chunks gives hbar at the chunk's
// end; pass B walks the 8-step sub-chunks backwards, recomputing their states
// into registers, and forms dx, ddelta, dA, dB, dC, dh0.  Sums over channels
// (dB, dC) and over batch and time (dA) are reduced in a fixed order: warp
// transpose-reduce, per-block partials, then a small reduction kernel.
#include <cuda_bf16.h>

#include <type_traits>

#include <algorithm>

#include "cla_internal.cuh"
#include "exp2_fma.cuh"
#include "mma_sync.cuh"

namespace cla {
namespace {

typedef __nv_bfloat16 bf16;

constexpr int kN = 16;        // state entries per channel
constexpr int kTc = 64;       // steps per chunk of the chunk-parallel kernels
constexpr int kCk = CLA_SELECTIVE_CKPT_CHUNK;  // steps between saved states (16)
static_assert(kTc % kCk == 0, "a chunk holds whole checkpoint intervals");
constexpr int kCh = 128;      // channels per block (forward)
constexpr int kChB = 64;      // channels per block (backward; measured: 5% faster than 128 there,
                              // 1.4% slower in the forward)
constexpr int kSubT = 8;      // backward sub-chunk length
constexpr float kLog2e = 1.4426950408889634f;


struct SelGeom {
    int B, D, n_chunks, n_cblk;
    long long T;
    long long n_ck;  // saved states per batch row: ceil(T / kCk)
};

struct SelWs {
    WsHeader *hdr;
    unsigned int *flags;  // per unit (chunk, b, cblk)
    float *agg;           // forward: [unit][17][kCh]; backward: [unit][32][kChB]
    float *incl;          // [unit][16][kCh or kChB]
    float *partB;         // [B][T][n_cblk][16]
    float *partC;
    float *partA;         // [B][n_chunks][D][16]
};

__device__ __forceinline__ size_t sel_unit(const SelGeom &g, int chunk, int b, int cblk) {
    return ((size_t)chunk * g.B + b) * g.n_cblk + cblk;
}

// ------------------------------------------------------------------ forward
struct SelFwdSmem {
    bf16 x[kTc][kCh];
    float d[kTc][kCh];
    float B[kTc][kN];
    float C[kTc][kN];
};

__global__ void __launch_bounds__(kCh)
sel_fwd_kernel(const bf16 *__restrict__ x, const float *__restrict__ delta, const float *__restrict__ A,
               const bf16 *__restrict__ Bm, const bf16 *__restrict__ Cm, const float *__restrict__ h0,
               float *__restrict__ y, float *__restrict__ hT, float *__restrict__ ckpt, SelGeom g, SelWs ws) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelFwdSmem &sm = *reinterpret_cast<SelFwdSmem *>(smem_raw);
    bf16(&s_x)[kTc][kCh] = sm.x;
    float(&s_d)[kTc][kCh] = sm.d;
    float(&s_B)[kTc][kN] = sm.B;
    float(&s_C)[kTc][kN] = sm.C;
    __shared__ unsigned int s_ticket, s_flag;

    const int tid = threadIdx.x;
    if (tid == 0) s_ticket = atomicAdd(&ws.hdr->ticket[0], 1u);
    __syncthreads();
    const unsigned int tk = s_ticket;
    const int per_chunk = g.B * g.n_cblk;
    const int chunk = (int)(tk / per_chunk);
    const int bi = (int)(tk % per_chunk) / g.n_cblk;
    const int cblk = (int)(tk % per_chunk) % g.n_cblk;
    const int c = cblk * kCh + tid;
    const bool cok = c < g.D;
    const long long t0 = (long long)chunk * kTc;
    const int L = (int)min((long long)kTc, g.T - t0);
    const size_t unit = sel_unit(g, chunk, bi, cblk);

    // stage the chunk: own channel column of x and delta, shared B_t and C_t rows
#pragma unroll 8
    for (int r = 0; r < kTc; ++r) {
        const bool ok = cok && r < L;
        const size_t idx = ((size_t)bi * g.T + t0 + r) * g.D + c;
        s_x[r][tid] = ok ? x[idx] : __float2bfloat16(0.f);
        s_d[r][tid] = ok ? __ldcs(delta + idx) : 0.f;
    }
    for (int i = tid; i < kTc * kN; i += kCh) {
        const int r = i / kN, n = i % kN;
        const bool ok = r < L;
        const size_t idx = ((size_t)bi * g.T + t0 + r) * kN + n;
        s_B[r][n] = ok ? __bfloat162float(Bm[idx]) : 0.f;
        s_C[r][n] = ok ? __bfloat162float(Cm[idx]) : 0.f;
    }
    __syncthreads();

    // state entries in pairs (n = 2j, 2j + 1) for the paired FP32 instructions
    constexpr int kJ = kN / 2;
    float A2[kN];
#pragma unroll
    for (int n = 0; n < kN; ++n) A2[n] = cok ? A[(size_t)c * kN + n] * kLog2e : 0.f;
    float2 A2p[kJ];
    float amax = 0.f;  // steps with |delta| * amax <= 126 need no clamp in 2^x
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        A2p[j] = make_float2(A2[2 * j], A2[2 * j + 1]);
        amax = fmaxf(amax, fmaxf(fabsf(A2[2 * j]), fabsf(A2[2 * j + 1])));
    }

    // phase 1: the chunk as one pair per n: (exp(A sum delta), Bagg)
    float2 Baggp[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) Baggp[j] = f2(0.f);
    float sumd = 0.f;
    for (int r = 0; r < L; ++r) {
        const float d = s_d[r][tid];
        const float dx = d * __bfloat162float(s_x[r][tid]);
        const float2 *Br = reinterpret_cast<const float2 *>(s_B[r]);
        auto step = [&](auto clamp) {
#pragma unroll
            for (int j = 0; j < kJ; ++j)
                Baggp[j] = __ffma2_rn(exp2_fma2<decltype(clamp)::value>(__fmul2_rn(f2(d), A2p[j])), Baggp[j],
                                      __fmul2_rn(f2(dx), Br[j]));
        };
        if (fabsf(d) * amax <= 126.f) step(std::false_type{});
        else step(std::true_type{});
        sumd += d;
    }
    float Bagg[kN];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        Bagg[2 * j] = Baggp[j].x;
        Bagg[2 * j + 1] = Baggp[j].y;
    }

    float hin[kN];
    if (chunk == 0) {
#pragma unroll
        for (int n = 0; n < kN; ++n) hin[n] = (h0 != nullptr && cok) ? h0[((size_t)bi * g.D + c) * kN + n] : 0.f;
    } else {
        float *ag = ws.agg + unit * (17 * kCh);
        __stcg(ag + tid, sumd);
#pragma unroll
        for (int n = 0; n < kN; ++n) __stcg(ag + (1 + n) * kCh + tid, Bagg[n]);
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(ws.flags + unit, 1u);
        float accS = 0.f, accB[kN];
#pragma unroll
        for (int n = 0; n < kN; ++n) accB[n] = 0.f;
        int j = chunk - 1;
        while (true) {
            const size_t up = sel_unit(g, j, bi, cblk);
            if (tid == 0) s_flag = wait_flag(ws.flags + up, ws.hdr, 20u);
            __syncthreads();
            const unsigned int f = s_flag;
            __syncthreads();
            if (f == 2u) {
                const float *ic = ws.incl + up * (kN * kCh);
#pragma unroll
                for (int n = 0; n < kN; ++n) hin[n] = fmaf(exp2_fma(A2[n] * accS), ld_cg(ic + n * kCh + tid), accB[n]);
                break;
            } else if (f == 1u) {
                const float *pa = ws.agg + up * (17 * kCh);
#pragma unroll
                for (int n = 0; n < kN; ++n) accB[n] = fmaf(exp2_fma(A2[n] * accS), ld_cg(pa + (1 + n) * kCh + tid), accB[n]);
                accS += ld_cg(pa + tid);
                if (--j < 0) {
#pragma unroll
                    for (int n = 0; n < kN; ++n) {
                        const float s0 = (h0 != nullptr && cok) ? h0[((size_t)bi * g.D + c) * kN + n] : 0.f;
                        hin[n] = fmaf(exp2_fma(A2[n] * accS), s0, accB[n]);
                    }
                    break;
                }
            } else {
#pragma unroll
                for (int n = 0; n < kN; ++n) hin[n] = 0.f;
                break;
            }
        }
    }
    {
        float *ic = ws.incl + unit * (kN * kCh);
#pragma unroll
        for (int n = 0; n < kN; ++n) __stcg(ic + n * kCh + tid, fmaf(exp2_fma(A2[n] * sumd), hin[n], Bagg[n]));
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(ws.flags + unit, 2u);
    }
    // phase 2: re-run from the true incoming state; write y once, and the state entering
    // every kCk-step interval for the backward
    float2 hp[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) hp[j] = make_float2(hin[2 * j], hin[2 * j + 1]);
    for (int r = 0; r < L; ++r) {
        if (ckpt != nullptr && cok && (r % kCk) == 0) {
            float4 *ck = reinterpret_cast<float4 *>(ckpt + (((size_t)bi * g.n_ck + (t0 + r) / kCk) * g.D + c) * kN);
#pragma unroll
            for (int q = 0; q < kN / 4; ++q)
                ck[q] = make_float4(hp[2 * q].x, hp[2 * q].y, hp[2 * q + 1].x, hp[2 * q + 1].y);
        }
        const float d = s_d[r][tid];
        const float dx = d * __bfloat162float(s_x[r][tid]);
        const float2 *Br = reinterpret_cast<const float2 *>(s_B[r]);
        const float2 *Cr = reinterpret_cast<const float2 *>(s_C[r]);
        float2 acc = f2(0.f);  // even and odd entries summed separately, then added
        auto step = [&](auto clamp) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                hp[j] = __ffma2_rn(exp2_fma2<decltype(clamp)::value>(__fmul2_rn(f2(d), A2p[j])), hp[j],
                                   __fmul2_rn(f2(dx), Br[j]));
                acc = __ffma2_rn(Cr[j], hp[j], acc);
            }
        };
        if (fabsf(d) * amax <= 126.f) step(std::false_type{});
        else step(std::true_type{});
        if (cok) __stcs(y + ((size_t)bi * g.T + t0 + r) * g.D + c, acc.x + acc.y);
    }
    if (hT != nullptr && cok && chunk == g.n_chunks - 1) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            hT[((size_t)bi * g.D + c) * kN + 2 * j] = hp[j].x;
            hT[((size_t)bi * g.D + c) * kN + 2 * j + 1] = hp[j].y;
        }
    }
}

// ------------------------------------------------- forward, one walk per channel
// With many channels (B * D) the chunk look-back is not needed to fill the GPU,
// and it costs a second evaluation of every decay (phase 1 folds a chunk, phase 2
// re-runs it).  This kernel walks each channel's whole sequence once.  A block
// owns 8 channels of one batch row; LANES lanes of a warp share a channel, lane
// LANES j + q holding state entries (16 / LANES) q.. of channel j.  Inputs are
// staged 64 steps at a time by cp.async (two buffers); a pass over each staged
// tile turns it into fp32 (delta, delta x) pairs per channel and fp32
// (B_n, B_n+1, C_n, C_n+1) quadruples per entry pair.  y_t sums a channel's 16
// entries over its lanes, LANES steps at a time: after the exchange lane q holds
// step q's sum.
constexpr int kSqCh = 8;                  // channels per block
constexpr int kSqTile = 64;               // steps per staged tile
static_assert(kSqTile % kCk == 0 && kCk % 8 == 0, "checkpoints fall on whole step groups of a tile");

struct SelSeqSmem {
    float d[2][kSqTile][kSqCh];       // staged delta
    bf16 x[2][kSqTile][kSqCh];        // staged x
    bf16 B[2][kSqTile][kN];           // staged B_t, C_t rows
    bf16 C[2][kSqTile][kN];
    float2 ddx[kSqTile][kSqCh];       // (delta, delta x) of the tile being walked
    float4 bc[kSqTile][kN / 2];       // (B_2p, B_2p+1, C_2p, C_2p+1) of the tile being walked
    // per channel j: lane q's y terms of 8 steps at [j][12 q + u] (rows of 104 floats: the
    // column sums read 8 lanes' rows without bank conflicts)
    float yx[kSqCh][104];
};

struct SelSeqGeom {
    int B, D;
    long long T, n_ck;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <int NT>
__device__ __forceinline__ void sel_seq_stage(SelSeqSmem &sm, int buf, const bf16 *x, const float *delta,
                                              const bf16 *Bm, const bf16 *Cm, const SelSeqGeom &g, int bi, int c0,
                                              long long t0, int tid) {
    const int L = (int)min((long long)kSqTile, g.T - t0);
    const size_t row0 = (size_t)bi * g.T + t0;
#pragma unroll
    for (int i = tid; i < kSqTile * 2; i += NT) {  // delta: 64 rows x two 16-byte pieces
        const int r = i >> 1, h = i & 1;
        if (r < L) cp_async16(smem_u32(&sm.d[buf][r][4 * h]), delta + (row0 + r) * g.D + c0 + 4 * h, 16u);
    }
#pragma unroll
    for (int r = tid; r < kSqTile; r += NT)  // x: 64 rows x one 16-byte piece
        if (r < L) cp_async16(smem_u32(&sm.x[buf][r][0]), x + (row0 + r) * g.D + c0, 16u);
#pragma unroll
    for (int i = tid; i < kSqTile * 2; i += NT) {  // B_t, C_t: 64 rows x two 16-byte pieces each
        const int r = i >> 1, h = i & 1;
        if (r < L) {
            cp_async16(smem_u32(&sm.B[buf][r][8 * h]), Bm + (row0 + r) * kN + 8 * h, 16u);
            cp_async16(smem_u32(&sm.C[buf][r][8 * h]), Cm + (row0 + r) * kN + 8 * h, 16u);
        }
    }
    cp_async_commit();
}

// Converts staged tile `buf` (rows past the sequence's end become delta = 0, which
// makes the step the identity: a = 1, b = 0) and returns whether every step of it
// satisfies |delta| * amax <= 126 (then 2^x needs no clamp).
template <int NT>
__device__ __forceinline__ bool sel_seq_convert(SelSeqSmem &sm, int buf, int L, float amax, int tid) {
    bool ok = true;
#pragma unroll
    for (int i = tid; i < kSqTile * kSqCh; i += NT) {
        const int r = i / kSqCh, cc = i % kSqCh;
        const float d = r < L ? sm.d[buf][r][cc] : 0.f;
        const float xv = r < L ? __bfloat162float(sm.x[buf][r][cc]) : 0.f;
        sm.ddx[r][cc] = make_float2(d, d * xv);
        ok = ok && (fabsf(d) * amax <= 126.f);
    }
    const uint32_t *Bw = reinterpret_cast<const uint32_t *>(sm.B[buf]);
    const uint32_t *Cw = reinterpret_cast<const uint32_t *>(sm.C[buf]);
    float4 *bc = &sm.bc[0][0];
#pragma unroll
    for (int i = tid; i < kSqTile * kN / 2; i += NT) {
        const int r = i / (kN / 2);
        const uint32_t bw = r < L ? Bw[i] : 0u, cw = r < L ? Cw[i] : 0u;
        bc[i] = make_float4(bf16_lo(bw), bf16_hi(bw), bf16_lo(cw), bf16_hi(cw));
    }
    return __syncthreads_and(ok) != 0;
}

template <int LANES>
__global__ void __launch_bounds__(kSqCh * LANES)
sel_fwd_seq_kernel(const bf16 *__restrict__ x, const float *__restrict__ delta, const float *__restrict__ A,
                   const bf16 *__restrict__ Bm, const bf16 *__restrict__ Cm, const float *__restrict__ h0,
                   float *__restrict__ y, float *__restrict__ hT, float *__restrict__ ckpt, SelSeqGeom g) {
    constexpr int NT = kSqCh * LANES;
    constexpr int NP = kN / LANES / 2;  // entry pairs per lane
    constexpr int G = LANES;            // steps per output exchange
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelSeqSmem &sm = *reinterpret_cast<SelSeqSmem *>(smem_raw);
    const int tid = threadIdx.x;
    const int bpr = g.D / kSqCh;  // blocks per batch row
    const int bi = (int)(blockIdx.x / bpr);
    const int c0 = (int)(blockIdx.x % bpr) * kSqCh;
    const int j = tid / LANES, q = tid % LANES;
    const int c = c0 + j, p0 = q * NP;  // this lane's first entry pair

    float2 A2p[NP];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        A2p[k] = make_float2(A[(size_t)c * kN + 2 * (p0 + k)] * kLog2e, A[(size_t)c * kN + 2 * (p0 + k) + 1] * kLog2e);
        amax = fmaxf(amax, fmaxf(fabsf(A2p[k].x), fabsf(A2p[k].y)));
    }
    {  // the block's largest |A| log2(e): the clamp test of a tile covers every channel of the block
        __shared__ float s_amax[NT / 32];
        s_amax[tid / 32] = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) amax = fmaxf(amax, s_amax[w]);
    }
    float2 h[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k)
        h[k] = h0 != nullptr ? make_float2(h0[((size_t)bi * g.D + c) * kN + 2 * (p0 + k)],
                                           h0[((size_t)bi * g.D + c) * kN + 2 * (p0 + k) + 1])
                             : f2(0.f);

    const int n_tiles = (int)((g.T + kSqTile - 1) / kSqTile);
    sel_seq_stage<NT>(sm, 0, x, delta, Bm, Cm, g, bi, c0, 0, tid);
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int buf = tile & 1;
        const long long t0 = (long long)tile * kSqTile;
        if (tile + 1 < n_tiles) {
            sel_seq_stage<NT>(sm, buf ^ 1, x, delta, Bm, Cm, g, bi, c0, t0 + kSqTile, tid);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // this tile's copies from every thread; the previous walk's reads done
        const int L = (int)min((long long)kSqTile, g.T - t0);
        const bool noclamp = sel_seq_convert<NT>(sm, buf, L, amax, tid);  // ends with a barrier
        auto walk = [&](auto clamp) {
            constexpr bool CL = decltype(clamp)::value;
#pragma unroll 2
            for (int s16 = 0; s16 < kSqTile; s16 += kCk) {
                if (ckpt != nullptr && t0 + s16 < g.T) {
                    float *ck = ckpt + (((size_t)bi * g.n_ck + (t0 + s16) / kCk) * g.D + c) * kN + 2 * p0;
                    if constexpr (NP == 2) {
                        *reinterpret_cast<float4 *>(ck) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
                    } else {
                        *reinterpret_cast<float2 *>(ck) = h[0];
                    }
                }
#pragma unroll
                for (int sg = 0; sg < kCk; sg += G) {
                    // the group's decays and inputs first (independent of the state), then
                    // the state recurrence through them
                    float2 a[G][NP], bx[G][NP], cc[G][NP];
#pragma unroll
                    for (int u = 0; u < G; ++u) {
                        const int r = s16 + sg + u;
                        const float2 dd = sm.ddx[r][j];
#pragma unroll
                        for (int k = 0; k < NP; ++k) {
                            const float4 bcv = sm.bc[r][p0 + k];
                            a[u][k] = exp2_fma2<CL>(__fmul2_rn(f2(dd.x), A2p[k]));
                            bx[u][k] = __fmul2_rn(f2(dd.y), make_float2(bcv.x, bcv.y));
                            cc[u][k] = make_float2(bcv.z, bcv.w);
                        }
                    }
                    float v[G];
#pragma unroll
                    for (int u = 0; u < G; ++u) {
                        float2 acc = f2(0.f);
#pragma unroll
                        for (int k = 0; k < NP; ++k) {
                            h[k] = __ffma2_rn(a[u][k], h[k], bx[u][k]);
                            acc = __ffma2_rn(cc[u][k], h[k], acc);
                        }
                        v[u] = acc.x + acc.y;
                    }
                    // sum over the channel's lanes through shared memory: lane q adds step q's
                    // terms of the channel's 8 lanes, in lane order
                    float yv;
                    if constexpr (G == 8) {
                        float *yr = sm.yx[j];
                        *reinterpret_cast<float4 *>(yr + 12 * q) = make_float4(v[0], v[1], v[2], v[3]);
                        *reinterpret_cast<float4 *>(yr + 12 * q + 4) = make_float4(v[4], v[5], v[6], v[7]);
                        __syncwarp();
                        yv = yr[q];
#pragma unroll
                        for (int i = 1; i < 8; ++i) yv += yr[12 * i + q];
                        __syncwarp();  // read before the next group's terms overwrite them
                    } else {  // 4 lanes: exchange by shuffles, lane q ends with step q's total
#pragma unroll
                        for (int m = G / 2; m >= 1; m >>= 1) {
                            const bool up = q & m;
#pragma unroll
                            for (int i = 0; i < m; ++i) {
                                const float keep = up ? v[i + m] : v[i];
                                const float send = up ? v[i] : v[i + m];
                                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                            }
                        }
                        yv = v[0];
                    }
                    const long long t = t0 + s16 + sg + q;
                    if (t < g.T) __stcs(y + ((size_t)bi * g.T + t) * g.D + c, yv);
                }
            }
        };
        if (noclamp) walk(std::false_type{});
        else walk(std::true_type{});
    }
    if (hT != nullptr) {
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            hT[((size_t)bi * g.D + c) * kN + 2 * (p0 + k)] = h[k].x;
            hT[((size_t)bi * g.D + c) * kN + 2 * (p0 + k) + 1] = h[k].y;
        }
    }
}

// ------------------------------------------------------------------ backward
constexpr int kBwdThreads = 2 * kChB;  // two threads per channel, 8 state entries each
constexpr int kNh = kN / 2;

struct SelBwdSmem {
    float x[kTc][kChB];
    float d[kTc + 1][kChB];  // row kTc: delta of the next chunk's first step
    float dy[kTc][kChB];
    float Bs[kTc][kN];
    float Cs[kTc][kN];
    float bnd[kTc / kSubT][kBwdThreads][kNh];  // state before every 8th step
    float red[kSubT][kBwdThreads / 32][2][kN];  // per-warp channel sums of dB, dC
};

// Sum of v[0..7] over the 16 lanes of this warp that share bit 0 of the lane
// index; returns the total for entry 4*b4 + 2*b3 + b2 (bits of the lane).
__device__ __forceinline__ float transpose_reduce8(float (&v)[kNh], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b4 ? v[j] : v[j + 4];
        const float keep = b4 ? v[j + 4] : v[j];
        w4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float w2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b3 ? w4[j] : w4[j + 2];
        const float keep = b3 ? w4[j + 2] : w4[j];
        w2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? w2[0] : w2[1];
    const float keep = b2 ? w2[1] : w2[0];
    float w1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
    return w1;
}

__global__ void __launch_bounds__(kBwdThreads)
sel_bwd_kernel(const bf16 *__restrict__ x, const float *__restrict__ delta, const float *__restrict__ A,
               const bf16 *__restrict__ Bm, const bf16 *__restrict__ Cm, const float *__restrict__ ckpt,
               const float *__restrict__ dy, const float *__restrict__ dhT, float *__restrict__ dx,
               float *__restrict__ ddelta, float *__restrict__ dh0, SelGeom g, SelWs ws) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelBwdSmem &sm = *reinterpret_cast<SelBwdSmem *>(smem_raw);
    __shared__ unsigned int s_ticket, s_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_ticket = atomicAdd(&ws.hdr->ticket[1], 1u);
    __syncthreads();
    const unsigned int tk = s_ticket;
    const int per_chunk = g.B * g.n_cblk;
    const int chunk = g.n_chunks - 1 - (int)(tk / per_chunk);
    const int bi = (int)(tk % per_chunk) / g.n_cblk;
    const int cblk = (int)(tk % per_chunk) % g.n_cblk;
    const int cl = tid >> 1, ng = tid & 1, n0 = ng * kNh;
    const int c = cblk * kChB + cl;
    const bool cok = c < g.D;
    const long long t0 = (long long)chunk * kTc;
    const int L = (int)min((long long)kTc, g.T - t0);
    const bool last = chunk == g.n_chunks - 1;
    const size_t unit = sel_unit(g, chunk, bi, cblk);

    for (int i = tid; i < kTc * kChB; i += kBwdThreads) {
        const int r = i / kChB, cc = i % kChB;
        const int ch = cblk * kChB + cc;
        const bool ok = ch < g.D && r < L;
        const size_t idx = ((size_t)bi * g.T + t0 + r) * g.D + ch;
        sm.x[r][cc] = ok ? __bfloat162float(x[idx]) : 0.f;
        sm.d[r][cc] = ok ? delta[idx] : 0.f;
        sm.dy[r][cc] = ok ? __ldcs(dy + idx) : 0.f;
    }
    for (int cc = tid; cc < kChB; cc += kBwdThreads) {
        const int ch = cblk * kChB + cc;
        sm.d[kTc][cc] = (!last && ch < g.D) ? delta[((size_t)bi * g.T + t0 + kTc) * g.D + ch] : 0.f;
    }
    for (int i = tid; i < kTc * kN; i += kBwdThreads) {
        const int r = i / kN, n = i % kN;
        const bool ok = r < L;
        const size_t idx = ((size_t)bi * g.T + t0 + r) * kN + n;
        sm.Bs[r][n] = ok ? __bfloat162float(Bm[idx]) : 0.f;
        sm.Cs[r][n] = ok ? __bfloat162float(Cm[idx]) : 0.f;
    }
    __syncthreads();

    float A2[kNh], Ar[kNh];
#pragma unroll
    for (int n = 0; n < kNh; ++n) {
        Ar[n] = cok ? A[(size_t)c * kN + n0 + n] : 0.f;
        A2[n] = Ar[n] * kLog2e;
    }
    // state entries in pairs (n0 + 2j, n0 + 2j + 1) for the paired FP32 instructions
    constexpr int kJh = kNh / 2;
    float2 A2p[kJh], Arp[kJh];
#pragma unroll
    for (int j = 0; j < kJh; ++j) {
        A2p[j] = make_float2(A2[2 * j], A2[2 * j + 1]);
        Arp[j] = make_float2(Ar[2 * j], Ar[2 * j + 1]);
    }
    // pass A: states (every 8th kept) and the adjoint pair of the chunk
    float P[kNh], Bg[kNh];
    {
        const float *ck = ckpt + (((size_t)bi * g.n_ck + (long long)chunk * (kTc / kCk)) * g.D + (cok ? c : 0)) * kN + n0;
        float2 hq[kJh], Pq[kJh], Bq[kJh];
#pragma unroll
        for (int j = 0; j < kJh; ++j) {
            hq[j] = cok ? make_float2(ck[2 * j], ck[2 * j + 1]) : f2(0.f);
            Pq[j] = f2(1.f);
            Bq[j] = f2(0.f);
        }
        for (int r = 0; r < L; ++r) {
            if ((r % kSubT) == 0) {
                float2 *bd = reinterpret_cast<float2 *>(sm.bnd[r / kSubT][tid]);
#pragma unroll
                for (int j = 0; j < kJh; ++j) bd[j] = hq[j];
            }
            const float d = sm.d[r][cl];
            const float dxv = d * sm.x[r][cl];
            const float gy = sm.dy[r][cl];
            const float2 *Cr = reinterpret_cast<const float2 *>(&sm.Cs[r][n0]);
            const float2 *Br = reinterpret_cast<const float2 *>(&sm.Bs[r][n0]);
#pragma unroll
            for (int j = 0; j < kJh; ++j) {
                const float2 a = exp2_fma2(__fmul2_rn(f2(d), A2p[j]));
                if (r > 0) Pq[j] = __fmul2_rn(Pq[j], a);
                Bq[j] = __ffma2_rn(Pq[j], __fmul2_rn(Cr[j], f2(gy)), Bq[j]);
                hq[j] = __ffma2_rn(a, hq[j], __fmul2_rn(f2(dxv), Br[j]));
            }
        }
#pragma unroll
        for (int j = 0; j < kJh; ++j) {
            P[2 * j] = Pq[j].x;
            P[2 * j + 1] = Pq[j].y;
            Bg[2 * j] = Bq[j].x;
            Bg[2 * j + 1] = Bq[j].y;
        }
    }
    float aend[kNh], Ag[kNh];
#pragma unroll
    for (int n = 0; n < kNh; ++n) {
        aend[n] = last ? 1.f : exp2_fma(sm.d[kTc][cl] * A2[n]);
        Ag[n] = P[n] * aend[n];
    }
    // look-back toward later chunks for hbar at the chunk's end
    float hb[kNh];
    if (last) {
#pragma unroll
        for (int n = 0; n < kNh; ++n) hb[n] = (dhT != nullptr && cok) ? dhT[((size_t)bi * g.D + c) * kN + n0 + n] : 0.f;
    } else {
        float *ag = ws.agg + unit * (32 * kChB);
#pragma unroll
        for (int n = 0; n < kNh; ++n) {
            __stcg(ag + (n0 + n) * kChB + cl, Ag[n]);
            __stcg(ag + (16 + n0 + n) * kChB + cl, Bg[n]);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(ws.flags + unit, 1u);
        float accA[kNh], accB[kNh];
#pragma unroll
        for (int n = 0; n < kNh; ++n) { accA[n] = 1.f; accB[n] = 0.f; }
        int j = chunk + 1;
        while (true) {
            const size_t up = sel_unit(g, j, bi, cblk);
            if (tid == 0) s_flag = wait_flag(ws.flags + up, ws.hdr, 21u);
            __syncthreads();
            const unsigned int f = s_flag;
            __syncthreads();
            if (f == 2u) {
                const float *ic = ws.incl + up * (kN * kChB);
#pragma unroll
                for (int n = 0; n < kNh; ++n) hb[n] = fmaf(accA[n], ld_cg(ic + (n0 + n) * kChB + cl), accB[n]);
                break;
            } else if (f == 1u) {
                const float *pa = ws.agg + up * (32 * kChB);
#pragma unroll
                for (int n = 0; n < kNh; ++n) {
                    accB[n] = fmaf(accA[n], ld_cg(pa + (16 + n0 + n) * kChB + cl), accB[n]);
                    accA[n] *= ld_cg(pa + (n0 + n) * kChB + cl);
                }
                if (++j >= g.n_chunks) {
#pragma unroll
                    for (int n = 0; n < kNh; ++n) {
                        const float s = (dhT != nullptr && cok) ? dhT[((size_t)bi * g.D + c) * kN + n0 + n] : 0.f;
                        hb[n] = fmaf(accA[n], s, accB[n]);
                    }
                    break;
                }
            } else {
#pragma unroll
                for (int n = 0; n < kNh; ++n) hb[n] = 0.f;
                break;
            }
        }
    }
    {
        float *ic = ws.incl + unit * (kN * kChB);
#pragma unroll
        for (int n = 0; n < kNh; ++n) __stcg(ic + (n0 + n) * kChB + cl, fmaf(Ag[n], hb[n], Bg[n]));
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release(ws.flags + unit, 2u);
    }

    // pass B: sub-chunks from last to first
    float2 anext[kJh], dA_acc[kJh], hbq[kJh];
#pragma unroll
    for (int j = 0; j < kJh; ++j) {
        anext[j] = make_float2(aend[2 * j], aend[2 * j + 1]);
        dA_acc[j] = f2(0.f);
        hbq[j] = make_float2(hb[2 * j], hb[2 * j + 1]);
    }
    const int nsub = (L + kSubT - 1) / kSubT;
    for (int k = nsub - 1; k >= 0; --k) {
        float2 hs[kSubT][kJh], as[kSubT][kJh], hstart[kJh], hq[kJh];
        {
            const float2 *bd = reinterpret_cast<const float2 *>(sm.bnd[k][tid]);
#pragma unroll
            for (int j = 0; j < kJh; ++j) {
                hstart[j] = bd[j];
                hq[j] = hstart[j];
            }
        }
#pragma unroll
        for (int i = 0; i < kSubT; ++i) {
            const int r = k * kSubT + i;
            const bool ok = r < L;
            const float d = ok ? sm.d[r][cl] : 0.f;
            const float dxv = d * (ok ? sm.x[r][cl] : 0.f);
            const float2 *Br = reinterpret_cast<const float2 *>(&sm.Bs[ok ? r : 0][n0]);
#pragma unroll
            for (int j = 0; j < kJh; ++j) {
                as[i][j] = exp2_fma2(__fmul2_rn(f2(d), A2p[j]));
                if (ok) hq[j] = __ffma2_rn(as[i][j], hq[j], __fmul2_rn(f2(dxv), Br[j]));
                hs[i][j] = hq[j];
            }
        }
#pragma unroll
        for (int i = kSubT - 1; i >= 0; --i) {
            const int r = k * kSubT + i;
            float vB[kNh], vC[kNh];
            if (r < L) {
                const float d = sm.d[r][cl], xv = sm.x[r][cl], gy = sm.dy[r][cl];
                const float2 *Br = reinterpret_cast<const float2 *>(&sm.Bs[r][n0]);
                const float2 *Cr = reinterpret_cast<const float2 *>(&sm.Cs[r][n0]);
                float2 sx2 = f2(0.f), sd2 = f2(0.f);  // even and odd entries, added at the end
#pragma unroll
                for (int j = 0; j < kJh; ++j) {
                    const float2 Bn = Br[j], Cn = Cr[j];
                    hbq[j] = __ffma2_rn(anext[j], hbq[j], __fmul2_rn(Cn, f2(gy)));
                    const float2 a = as[i][j];
                    const float2 hp = (i > 0) ? hs[i - 1][j] : hstart[j];
                    const float2 ga = __fmul2_rn(__fmul2_rn(hbq[j], hp), a);  // dL/da_t * a_t
                    sx2 = __ffma2_rn(hbq[j], Bn, sx2);
                    sd2 = __ffma2_rn(ga, Arp[j], __ffma2_rn(hbq[j], __fmul2_rn(Bn, f2(xv)), sd2));
                    dA_acc[j] = __ffma2_rn(ga, f2(d), dA_acc[j]);
                    const float2 vb = __fmul2_rn(__fmul2_rn(hbq[j], f2(d)), f2(xv));
                    const float2 vc = __fmul2_rn(f2(gy), hs[i][j]);
                    vB[2 * j] = vb.x;
                    vB[2 * j + 1] = vb.y;
                    vC[2 * j] = vc.x;
                    vC[2 * j + 1] = vc.y;
                    anext[j] = a;
                }
                float sx = sx2.x + sx2.y, sd = sd2.x + sd2.y;
                sx += __shfl_xor_sync(0xffffffffu, sx, 1);
                sd += __shfl_xor_sync(0xffffffffu, sd, 1);
                if (ng == 0 && cok) {
                    const size_t idx = ((size_t)bi * g.T + t0 + r) * g.D + c;
                    __stcs(dx + idx, sx * d);
                    __stcs(ddelta + idx, sd);
                }
                if (r == 0 && chunk == 0 && dh0 != nullptr && cok) {
#pragma unroll
                    for (int j = 0; j < kJh; ++j) {
                        const float2 v = __fmul2_rn(anext[j], hbq[j]);
                        dh0[((size_t)bi * g.D + c) * kN + n0 + 2 * j] = v.x;
                        dh0[((size_t)bi * g.D + c) * kN + n0 + 2 * j + 1] = v.y;
                    }
                }
            } else {
#pragma unroll
                for (int n = 0; n < kNh; ++n) { vB[n] = 0.f; vC[n] = 0.f; }
            }
            if (!cok) {
#pragma unroll
                for (int n = 0; n < kNh; ++n) { vB[n] = 0.f; vC[n] = 0.f; }
            }
            // channel sums of this warp's 16 channels; lane keeps entry e of its half
            const float sB = transpose_reduce8(vB, lane);
            const float sC = transpose_reduce8(vC, lane);
            if ((lane & 2) == 0) {
                const int e = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                sm.red[i][warp][0][n0 + e] = sB;
                sm.red[i][warp][1][n0 + e] = sC;
            }
        }
        __syncthreads();
        // block partials over the block's channels, in warp order
        for (int idx = tid; idx < kSubT * 32; idx += kBwdThreads) {
            const int i = idx >> 5, w = idx & 31;  // 8 steps x (2 quantities x 16 entries)
            const int q = w >> 4, n = w & 15;
            const int r = k * kSubT + i;
            if (r < L) {
                float s = 0.f;
#pragma unroll
                for (int ww = 0; ww < kBwdThreads / 32; ++ww) s += sm.red[i][ww][q][n];
                float *dst = (q == 0 ? ws.partB : ws.partC);
                dst[(((size_t)bi * g.T + t0 + r) * g.n_cblk + cblk) * kN + n] = s;
            }
        }
        __syncthreads();
    }
    if (ws.partA != nullptr && cok) {
        float *pa = ws.partA + (((size_t)bi * g.n_chunks + chunk) * g.D + c) * kN + n0;
#pragma unroll
        for (int j = 0; j < kJh; ++j) {
            pa[2 * j] = dA_acc[j].x;
            pa[2 * j + 1] = dA_acc[j].y;
        }
    }
}

// ------------------------------------------------ backward, one walk per channel
// The counterpart of sel_fwd_seq_kernel: with many channels each block walks its 8
// channels of one batch row from the last step to the first, so no look-back over
// later chunks is needed, and the saved states (one every kCk = 16 steps) let every
// 16-step interval be recomputed forward once -- decays and states kept in registers
// -- before the adjoint runs back through it: one decay evaluation per state update
// (the chunk-parallel backward needs two).  Inputs are staged 32 steps at a time by
// cp.async (two buffers) and converted to fp32 (delta, delta x, x, dy) per channel and
// (B, C) per entry pair.  The sums over a channel's entries (dx, ddelta) and over the
// block's channels (dB, dC) go through shared memory every 8 steps, in a fixed order;
// the block's dB, dC partials are summed over blocks by sel_reduce_bc_kernel.
constexpr int kSbTile = 32;  // steps per staged tile
constexpr int kSbGrp = 8;    // steps per exchange of the sums
static_assert(kSbTile % kCk == 0 && kCk % kSbGrp == 0, "tiles hold whole recompute intervals");

template <int CH>  // channels per block
struct SelSeqBwdSmem {
    float d[2][kSbTile][CH];      // staged delta, x, dy, B_t, C_t
    bf16 x[2][kSbTile][CH];
    float dy[2][kSbTile][CH];
    bf16 B[2][kSbTile][kN];
    bf16 C[2][kSbTile][kN];
    float4 dxy[kSbTile][CH];      // (delta, delta x, x, dy) of the tile being walked
    float4 bc[kSbTile][kN / 2];   // (B_2p, B_2p+1, C_2p, C_2p+1)
    float4 rbc[kSbGrp][CH][kN / 2];  // per step: dB, dC terms of channel j, entry pair p
    float2 rxd[kSbGrp][CH][8 + 1];   // per step: channel j's lane q terms of dx / delta, ddelta
                                     // (rows padded: the channel sums read them across rows)
};

template <int CH>
__device__ __forceinline__ void sel_seqb_stage(SelSeqBwdSmem<CH> &sm, int buf, const bf16 *x, const float *delta,
                                               const float *dy, const bf16 *Bm, const bf16 *Cm,
                                               const SelSeqGeom &g, int bi, int c0, long long t0, int tid) {
    constexpr int NT = CH * 8;
    constexpr int PF = CH / 4, PX = CH / 8;  // 16-byte pieces per row of delta / dy and of x
    const int L = (int)min((long long)kSbTile, g.T - t0);
    const size_t row0 = (size_t)bi * g.T + t0;
#pragma unroll
    for (int i = tid; i < kSbTile * PF; i += NT) {  // delta, dy
        const int r = i / PF, h = i % PF;
        if (r < L) {
            cp_async16(smem_u32(&sm.d[buf][r][4 * h]), delta + (row0 + r) * g.D + c0 + 4 * h, 16u);
            cp_async16(smem_u32(&sm.dy[buf][r][4 * h]), dy + (row0 + r) * g.D + c0 + 4 * h, 16u);
        }
    }
#pragma unroll
    for (int i = tid; i < kSbTile * PX; i += NT) {  // x
        const int r = i / PX, h = i % PX;
        if (r < L) cp_async16(smem_u32(&sm.x[buf][r][8 * h]), x + (row0 + r) * g.D + c0 + 8 * h, 16u);
    }
#pragma unroll
    for (int i = tid; i < kSbTile * 2; i += NT) {  // B_t, C_t: two 16-byte pieces each per row
        const int r = i >> 1, h = i & 1;
        if (r < L) {
            cp_async16(smem_u32(&sm.B[buf][r][8 * h]), Bm + (row0 + r) * kN + 8 * h, 16u);
            cp_async16(smem_u32(&sm.C[buf][r][8 * h]), Cm + (row0 + r) * kN + 8 * h, 16u);
        }
    }
    cp_async_commit();
}

// As sel_seq_convert: rows past the end become delta = dy = x = 0 and B = C = 0, which
// leaves the adjoint unchanged through them and adds nothing to any gradient.
template <int CH>
__device__ __forceinline__ bool sel_seqb_convert(SelSeqBwdSmem<CH> &sm, int buf, int L, float amax, int tid) {
    constexpr int NT = CH * 8;
    bool ok = true;
#pragma unroll
    for (int i = tid; i < kSbTile * CH; i += NT) {
        const int r = i / CH, cc = i % CH;
        const float d = r < L ? sm.d[buf][r][cc] : 0.f;
        const float xv = r < L ? __bfloat162float(sm.x[buf][r][cc]) : 0.f;
        const float g = r < L ? sm.dy[buf][r][cc] : 0.f;
        sm.dxy[r][cc] = make_float4(d, d * xv, xv, g);
        ok = ok && (fabsf(d) * amax <= 126.f);
    }
    const uint32_t *Bw = reinterpret_cast<const uint32_t *>(sm.B[buf]);
    const uint32_t *Cw = reinterpret_cast<const uint32_t *>(sm.C[buf]);
    float4 *bc = &sm.bc[0][0];
#pragma unroll
    for (int i = tid; i < kSbTile * kN / 2; i += NT) {
        const int r = i / (kN / 2);
        const uint32_t bw = r < L ? Bw[i] : 0u, cw = r < L ? Cw[i] : 0u;
        bc[i] = make_float4(bf16_lo(bw), bf16_hi(bw), bf16_lo(cw), bf16_hi(cw));
    }
    return __syncthreads_and(ok) != 0;
}

// 8 lanes per channel (entries 2q, 2q + 1 on lane q), CH channels per block (more
// channels per block: fewer dB, dC partials to write and sum over blocks).
// Blocks per SM: 7 of 8 channels or 4 of 16 (shared memory allows 7 and 4; registers
// are capped at 128 per thread for them), so that every block of the workload's grid is
// resident at once.
template <int CH>
__global__ void __launch_bounds__(CH * 8, CH == 8 ? 7 : 4)
sel_bwd_seq_kernel(const bf16 *__restrict__ x, const float *__restrict__ delta, const float *__restrict__ A,
                   const bf16 *__restrict__ Bm, const bf16 *__restrict__ Cm, const float *__restrict__ ckpt,
                   const float *__restrict__ dy, const float *__restrict__ dhT, float *__restrict__ dx,
                   float *__restrict__ ddelta, float *__restrict__ dh0, float *__restrict__ partB,
                   float *__restrict__ partC, float *__restrict__ partA, SelSeqGeom g) {
    constexpr int NT = CH * 8;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelSeqBwdSmem<CH> &sm = *reinterpret_cast<SelSeqBwdSmem<CH> *>(smem_raw);
    const int tid = threadIdx.x;
    const int bpr = g.D / CH;  // blocks per batch row
    const int bi = (int)(blockIdx.x / bpr), blk = (int)(blockIdx.x % bpr);
    const int c0 = blk * CH;
    const int j = tid >> 3, q = tid & 7;
    const int c = c0 + j;

    const float2 Ar = make_float2(A[(size_t)c * kN + 2 * q], A[(size_t)c * kN + 2 * q + 1]);
    const float2 A2 = make_float2(Ar.x * kLog2e, Ar.y * kLog2e);
    float amax = fmaxf(fabsf(A2.x), fabsf(A2.y));
    {  // the block's largest |A| log2(e), as in the forward
        __shared__ float s_amax[NT / 32];
        s_amax[tid / 32] = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) amax = fmaxf(amax, s_amax[w]);
    }
    const size_t sidx = ((size_t)bi * g.D + c) * kN + 2 * q;  // this lane's entries in [B, D, N]
    float2 hb = dhT != nullptr ? make_float2(dhT[sidx], dhT[sidx + 1]) : f2(0.f);
    // dA over the whole walk: summed per 16-step interval, the interval sums added with
    // compensation (a plain running fp32 sum over thousands of steps drifts past 1e-5)
    float2 anext = f2(1.f), dA_acc = f2(0.f), dA_cmp = f2(0.f);

    const int n_tiles = (int)((g.T + kSbTile - 1) / kSbTile);
    // the saved state entering the interval walked next, loaded one interval ahead
    const float *ckc = ckpt + ((size_t)bi * g.n_ck * g.D + c) * kN + 2 * q;
    const size_t ck_stride = (size_t)g.D * kN;
    long long ck_next = g.n_ck - 1;
    float2 hin_next = *reinterpret_cast<const float2 *>(ckc + ck_next * ck_stride);
    sel_seqb_stage(sm, (n_tiles - 1) & 1, x, delta, dy, Bm, Cm, g, bi, c0, (long long)(n_tiles - 1) * kSbTile, tid);
    for (int tile = n_tiles - 1; tile >= 0; --tile) {
        const int buf = tile & 1;
        const long long t0 = (long long)tile * kSbTile;
        if (tile > 0) {
            sel_seqb_stage(sm, buf ^ 1, x, delta, dy, Bm, Cm, g, bi, c0, t0 - kSbTile, tid);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // this tile's copies from every thread; the previous tile's reads done
        const int L = (int)min((long long)kSbTile, g.T - t0);
        const bool noclamp = sel_seqb_convert(sm, buf, L, amax, tid);  // ends with a barrier
        auto walk = [&](auto clamp) {
            constexpr bool CL = decltype(clamp)::value;
#pragma unroll 1
            for (int s = kSbTile - kCk; s >= 0; s -= kCk) {
                if (t0 + s >= g.T) continue;  // an interval wholly past the end (uniform)
                // recompute the interval's decays and states from the saved state
                const float2 hin = hin_next;  // intervals are walked in order: this is (t0 + s) / kCk
                if (--ck_next >= 0) hin_next = *reinterpret_cast<const float2 *>(ckc + ck_next * ck_stride);
                float2 as[kCk], hs[kCk];
                {
                    float2 h = hin;
#pragma unroll
                    for (int u = 0; u < kCk; ++u) {
                        const float4 v = sm.dxy[s + u][j];
                        const float4 b = sm.bc[s + u][q];
                        as[u] = exp2_fma2<CL>(__fmul2_rn(f2(v.x), A2));
                        h = __ffma2_rn(as[u], h, __fmul2_rn(f2(v.y), make_float2(b.x, b.y)));
                        hs[u] = h;
                    }
                }
                // the adjoint back through the interval, 8 steps per exchange of the sums
                float2 dA_loc = f2(0.f);
#pragma unroll
                for (int gi = kCk / kSbGrp - 1; gi >= 0; --gi) {
#pragma unroll
                    for (int uu = kSbGrp - 1; uu >= 0; --uu) {
                        const int u = gi * kSbGrp + uu, r = s + u;
                        const float4 v = sm.dxy[r][j];  // (delta, delta x, x, dy)
                        const float4 b = sm.bc[r][q];   // (B, B', C, C')
                        const float2 Bp = make_float2(b.x, b.y);
                        hb = __ffma2_rn(anext, hb, __fmul2_rn(make_float2(b.z, b.w), f2(v.w)));
                        const float2 a = as[u];
                        const float2 hp = u > 0 ? hs[u - 1] : hin;
                        const float2 ga = __fmul2_rn(__fmul2_rn(hb, hp), a);  // dL/da * a
                        const float2 sb = __fmul2_rn(hb, Bp);
                        const float sx = sb.x + sb.y;                        // sum_n hbar B
                        const float2 sd2 = __ffma2_rn(ga, Ar, __fmul2_rn(sb, f2(v.z)));
                        dA_loc = __ffma2_rn(ga, f2(v.x), dA_loc);
                        const float2 vb = __fmul2_rn(hb, f2(v.y));             // hbar delta x
                        const float2 vc = __fmul2_rn(hs[u], f2(v.w));          // dy h
                        anext = a;
                        sm.rbc[uu][j][q] = make_float4(vb.x, vb.y, vc.x, vc.y);
                        sm.rxd[uu][j][q] = make_float2(sx, sd2.x + sd2.y);
                        if (u == 0 && t0 + s == 0 && dh0 != nullptr) {  // step 0 of the sequence
                            const float2 v0 = __fmul2_rn(anext, hb);
                            dh0[sidx] = v0.x;
                            dh0[sidx + 1] = v0.y;
                        }
                    }
                    __syncthreads();
                    {  // thread (step uu, channel k): dx, ddelta summed over the channel's lanes
                        const int uu = tid / CH, k = tid % CH;
                        const long long t = t0 + s + gi * kSbGrp + uu;
                        float2 sxd = sm.rxd[uu][k][0];
#pragma unroll
                        for (int i = 1; i < 8; ++i) sxd = __fadd2_rn(sxd, sm.rxd[uu][k][i]);
                        if (t < g.T) {
                            const size_t oidx = ((size_t)bi * g.T + t) * g.D + c0 + k;
                            __stcs(dx + oidx, sxd.x * sm.dxy[s + gi * kSbGrp + uu][k].x);
                            __stcs(ddelta + oidx, sxd.y);
                        }
                    }
                    if (tid < kSbGrp * kN / 2) {  // thread (step uu, entry pair k): dB, dC in channel order
                        const int uu = tid >> 3, k = tid & 7;
                        const long long t = t0 + s + gi * kSbGrp + uu;
                        const float4 w0 = sm.rbc[uu][0][k];
                        float2 sb2 = make_float2(w0.x, w0.y), sc2 = make_float2(w0.z, w0.w);
#pragma unroll
                        for (int i = 1; i < CH; ++i) {
                            const float4 w = sm.rbc[uu][i][k];
                            sb2 = __fadd2_rn(sb2, make_float2(w.x, w.y));
                            sc2 = __fadd2_rn(sc2, make_float2(w.z, w.w));
                        }
                        if (t < g.T) {
                            const size_t pidx = (((size_t)bi * g.T + t) * bpr + blk) * kN + 2 * k;
                            *reinterpret_cast<float2 *>(partB + pidx) = sb2;
                            *reinterpret_cast<float2 *>(partC + pidx) = sc2;
                        }
                    }
                    __syncthreads();
                }
                {  // Kahan step: dA_acc + dA_loc, the rounding error kept in dA_cmp
                    const float2 yv = __fadd2_rn(dA_loc, make_float2(-dA_cmp.x, -dA_cmp.y));
                    const float2 tv = __fadd2_rn(dA_acc, yv);
                    dA_cmp = __fadd2_rn(__fadd2_rn(tv, make_float2(-dA_acc.x, -dA_acc.y)), make_float2(-yv.x, -yv.y));
                    dA_acc = tv;
                }
            }
        };
        if (noclamp) walk(std::false_type{});
        else walk(std::true_type{});
    }
    if (partA != nullptr) *reinterpret_cast<float2 *>(partA + sidx) = dA_acc;
}

// dB, dC: sums of the per-block partials, in block order.
__global__ void sel_reduce_bc_kernel(const float *__restrict__ partB, const float *__restrict__ partC,
                                     float *__restrict__ dB, float *__restrict__ dC, long long rows, int n_cblk) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (b, t, n)
    if (i >= rows * kN) return;
    const long long row = i / kN;
    const int n = (int)(i % kN);
    float sb = 0.f, sc = 0.f;
    for (int k = 0; k < n_cblk; ++k) {
        sb += partB[(row * n_cblk + k) * kN + n];
        sc += partC[(row * n_cblk + k) * kN + n];
    }
    dB[i] = sb;
    dC[i] = sc;
}

// dA[d][n]: sum over batch rows and chunks, in that order.
// dA[i] = sum over (b, chunk) of partA[b][chunk][i]: a block takes 32 consecutive i (one
// coalesced 128-byte row per (b, chunk)); its 8 warps split the (b, chunk) rows (warp w takes
// rows w, w + 8, ...) and add their sums in warp order, so the order is fixed.
constexpr int kRedAWarps = 8;
__global__ void __launch_bounds__(kRedAWarps * 32)
sel_reduce_a_kernel(const float *__restrict__ partA, float *__restrict__ dA, int B, int n_chunks, int D) {
    __shared__ float s_part[kRedAWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long n_i = (long long)D * kN;
    const long long i = (long long)blockIdx.x * 32 + lane;  // (d, n)
    const long long rows = (long long)B * n_chunks;
    float s = 0.f;
    if (i < n_i) {
        long long r = warp;
        // four rows in flight per thread
        for (; r + 3 * kRedAWarps < rows; r += 4 * kRedAWarps) {
            const float v0 = partA[r * n_i + i], v1 = partA[(r + kRedAWarps) * n_i + i];
            const float v2 = partA[(r + 2 * kRedAWarps) * n_i + i], v3 = partA[(r + 3 * kRedAWarps) * n_i + i];
            s += v0;
            s += v1;
            s += v2;
            s += v3;
        }
        for (; r < rows; r += kRedAWarps) s += partA[r * n_i + i];
    }
    s_part[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && i < n_i) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kRedAWarps; ++w) t += s_part[w][lane];
        dA[i] = t;
    }
}

// ------------------------------------------------------------------ host side
constexpr int kSqLanes = 8;  // lanes per channel (2 entries each): two warps per block
// The per-channel walks (sel_fwd_seq_kernel, sel_bwd_seq_kernel) are taken when their
// warps (one per 4 channels of a batch row) give every SM at least four, so that a
// walk's dependent steps overlap other warps' work; they need D a multiple of 8 and
// 16-byte aligned rows for their staged copies.
bool sel_walk_sizes(int64_t B, int64_t D) {
    if (D % kSqCh != 0 || D == 0) return false;
    const double blocks = (double)B * (double)(D / kSqCh);
    if (blocks >= 2147483648.0) return false;
    const double warps = blocks * kSqCh * kSqLanes / 32;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    return warps >= 4.0 * sms;
}
// Channels per block of the backward walk.  16 (half the dB, dC partials to write and sum)
// measured slower on the 4 x 8192 x 2048 workload: 2300 against 2192 us (4 blocks of 4 warps
// per SM against 7 of 2).
constexpr int kSbCh = 8;
bool sel_use_seq(bool walk_sizes, std::initializer_list<const void *> rows) {
    if (!walk_sizes) return false;
    for (const void *r : rows)
        if (!aligned16(r)) return false;
    return true;
}

struct SelPlan {
    SelGeom g, gb;  // forward and backward geometry (their channel blocks differ)
    bool walk;      // sizes for which the per-channel walks run (with aligned rows)
    size_t units;
    size_t off_flags, off_agg, off_incl, off_pB, off_pC, off_pA, total;
};

SelPlan sel_plan(int64_t B, int64_t T, int64_t D) {
    SelPlan p;
    p.g.B = (int)B;
    p.g.D = (int)D;
    p.g.T = T;
    p.g.n_chunks = (int)((T + kTc - 1) / kTc);
    p.g.n_ck = (T + kCk - 1) / kCk;
    p.g.n_cblk = (int)((D + kCh - 1) / kCh);
    p.gb = p.g;
    p.gb.n_cblk = (int)((D + kChB - 1) / kChB);
    p.walk = sel_walk_sizes(B, D);
    // dB, dC partials: one per channel block of the backward that runs
    const size_t n_part = std::max((size_t)p.gb.n_cblk, p.walk ? (size_t)(D / kSbCh) : (size_t)0);
    const size_t units_f = (size_t)p.g.n_chunks * B * p.g.n_cblk, units_b = (size_t)p.g.n_chunks * B * p.gb.n_cblk;
    p.units = units_f > units_b ? units_f : units_b;
    const size_t lanes = std::max(units_f * kCh, units_b * kChB);  // channel slots over all units
    p.off_flags = sizeof(WsHeader);
    p.off_agg = align_up(p.off_flags + p.units * 4, 256);
    p.off_incl = align_up(p.off_agg + lanes * 32 * 4, 256);
    p.off_pB = align_up(p.off_incl + lanes * kN * 4, 256);
    p.off_pC = align_up(p.off_pB + (size_t)B * T * n_part * kN * 4, 256);
    p.off_pA = align_up(p.off_pC + (size_t)B * T * n_part * kN * 4, 256);
    p.total = align_up(p.off_pA + (size_t)B * p.g.n_chunks * D * kN * 4, 256);
    return p;
}

SelWs sel_bind(const SelPlan &p, void *ws) {
    char *w = static_cast<char *>(ws);
    SelWs s;
    s.hdr = reinterpret_cast<WsHeader *>(w);
    s.flags = reinterpret_cast<unsigned int *>(w + p.off_flags);
    s.agg = reinterpret_cast<float *>(w + p.off_agg);
    s.incl = reinterpret_cast<float *>(w + p.off_incl);
    s.partB = reinterpret_cast<float *>(w + p.off_pB);
    s.partC = reinterpret_cast<float *>(w + p.off_pC);
    s.partA = reinterpret_cast<float *>(w + p.off_pA);
    return s;
}

// Non-negative sizes every kernel and plan of this file handles: the larger
// (backward) grid stays below 2^31 blocks.
bool sel_sizes_fit(int64_t B, int64_t T, int64_t D) {
    if (D > (1 << 24) || B > (1 << 20) || T > (1ll << 36)) return false;
    return product_below({(T + kTc - 1) / kTc, B, (D + kChB - 1) / kChB}, 2147483648.0);
}

// The one-walk-per-channel forward is taken when its warps (one per 4 channels of a
// batch row) give every SM at least four, so that a walk's dependent steps overlap
// other warps' work; it needs 16-byte aligned rows for its staged copies.
int sel_validate(const char *fn, int64_t B, int64_t T, int64_t D, int64_t N) {
    if (B < 0 || T < 0 || D < 0 || N < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (N != kN) return fail(CLA_ERR_UNSUPPORTED, "%s: N must be %d (got %lld)", fn, kN, (long long)N);
    if (!sel_sizes_fit(B, T, D)) return fail(CLA_ERR_UNSUPPORTED, "%s: size out of range for one launch", fn);
    return CLA_OK;
}

}  // namespace
}  // namespace cla

using namespace cla;

extern "C" size_t cla_selective_scan_workspace_size(int64_t B, int64_t T, int64_t D, int64_t N) {
    if (B < 0 || T < 0 || D < 0 || N != kN || !sel_sizes_fit(B, T, D)) return 0;
    return sel_plan(B, T, D).total;
}

extern "C" size_t cla_selective_scan_ckpt_elems(int64_t B, int64_t T, int64_t D, int64_t N) {
    if (B < 0 || T < 0 || D < 0 || N != kN || !sel_sizes_fit(B, T, D)) return 0;
    return (size_t)B * (size_t)((T + kCk - 1) / kCk) * (size_t)D * (size_t)N;
}

extern "C" int cla_selective_scan_fwd(const uint16_t *x, const float *delta, const float *A, const uint16_t *Bm,
                                      const uint16_t *Cm, const float *h0, float *y, float *hT, float *ckpt,
                                      int64_t B, int64_t T, int64_t D, int64_t N, void *ws, size_t ws_bytes,
                                      void *stream) {
    clear_error();
    const char *fn = "cla_selective_scan_fwd";
    int st = sel_validate(fn, B, T, D, N);
    if (st) return st;
    if (!aligned_or_null({delta, A, h0, y, hT}, 4) || !aligned_or_null({x, Bm, Cm}, 2))
        return fail(CLA_ERR_INVALID_ARG, "%s: tensors must be aligned to their element size", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return CLA_OK;
    if (T == 0) {
        if (hT) {
            const size_t by = sizeof(float) * B * D * N;
            if (h0) CLA_CUDA_TRY(cudaMemcpyAsync(hT, h0, by, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(hT, 0, by, s), fn);
        }
        return CLA_OK;
    }
    if (!x || !delta || !A || !Bm || !Cm || !y) return fail(CLA_ERR_INVALID_ARG, "%s: x, delta, A, Bm, Cm, y required", fn);
    if (!aligned16_or_null(ckpt)) return fail(CLA_ERR_INVALID_ARG, "%s: ckpt must be 16-byte aligned", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    const SelPlan p = sel_plan(B, T, D);
    if (ws_bytes < p.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, p.total);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.off_agg, s), fn);
    if (sel_use_seq(p.walk, {x, delta, Bm, Cm})) {
        // one-warp blocks: as many per SM as shared memory holds (all of it as shared memory)
        static std::atomic<unsigned long long> carve_set{0};
        st = set_smem_carveout_max(carve_set, reinterpret_cast<const void *>(sel_fwd_seq_kernel<kSqLanes>));
        if (st) return st;
        const SelSeqGeom sg{(int)B, (int)D, T, p.g.n_ck};
        const unsigned int grid = (unsigned int)(B * (D / kSqCh));
        sel_fwd_seq_kernel<kSqLanes><<<grid, kSqCh * kSqLanes, sizeof(SelSeqSmem), s>>>(
            reinterpret_cast<const bf16 *>(x), delta, A, reinterpret_cast<const bf16 *>(Bm),
            reinterpret_cast<const bf16 *>(Cm), h0, y, hT, ckpt, sg);
        return check_launch(fn);
    }
    const SelWs w = sel_bind(p, ws);
    static std::atomic<unsigned long long> smem_set{0};
    st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(sel_fwd_kernel), (int)sizeof(SelFwdSmem));
    if (st) return st;
    const unsigned int grid = (unsigned int)((size_t)p.g.n_chunks * B * p.g.n_cblk);
    sel_fwd_kernel<<<grid, kCh, sizeof(SelFwdSmem), s>>>(reinterpret_cast<const bf16 *>(x), delta, A, reinterpret_cast<const bf16 *>(Bm),
                                        reinterpret_cast<const bf16 *>(Cm), h0, y, hT, ckpt, p.g, w);
    return check_launch(fn);
}

extern "C" int cla_selective_scan_bwd(const uint16_t *x, const float *delta, const float *A, const uint16_t *Bm,
                                      const uint16_t *Cm, const float *h0, const float *ckpt, const float *dy,
                                      const float *dhT, float *dx, float *ddelta, float *dA, float *dB, float *dC,
                                      float *dh0, int64_t B, int64_t T, int64_t D, int64_t N, void *ws,
                                      size_t ws_bytes, void *stream) {
    clear_error();
    const char *fn = "cla_selective_scan_bwd";
    int st = sel_validate(fn, B, T, D, N);
    if (st) return st;
    (void)h0;  // the checkpoints already contain the initial state
    if (!aligned_or_null({delta, A, ckpt, dy, dhT, dx, ddelta, dA, dB, dC, dh0}, 4) ||
        !aligned_or_null({x, Bm, Cm}, 2))
        return fail(CLA_ERR_INVALID_ARG, "%s: tensors must be aligned to their element size", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) {
        if (dA && D > 0) CLA_CUDA_TRY(cudaMemsetAsync(dA, 0, sizeof(float) * D * N, s), fn);
        return CLA_OK;
    }
    if (T == 0) {
        if (dA) CLA_CUDA_TRY(cudaMemsetAsync(dA, 0, sizeof(float) * D * N, s), fn);
        if (dh0) {
            const size_t by = sizeof(float) * B * D * N;
            if (dhT) CLA_CUDA_TRY(cudaMemcpyAsync(dh0, dhT, by, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(dh0, 0, by, s), fn);
        }
        return CLA_OK;
    }
    if (!x || !delta || !A || !Bm || !Cm || !ckpt || !dy || !dx || !ddelta || !dB || !dC)
        return fail(CLA_ERR_INVALID_ARG, "%s: x, delta, A, Bm, Cm, ckpt, dy, dx, ddelta, dB, dC required", fn);
    if (!ws || !aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace NULL or unaligned", fn);
    const SelPlan p = sel_plan(B, T, D);
    if (ws_bytes < p.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, p.total);
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.off_agg, s), fn);
    SelWs w = sel_bind(p, ws);
    if (!dA) w.partA = nullptr;
    const long long rows = B * T;
    if (sel_use_seq(p.walk, {x, delta, dy, Bm, Cm})) {
        constexpr int CH = kSbCh;
        const SelSeqGeom sg{(int)B, (int)D, T, p.g.n_ck};
        const unsigned int grid = (unsigned int)(B * (D / CH));
        const void *fnp = reinterpret_cast<const void *>(sel_bwd_seq_kernel<CH>);
        static std::atomic<unsigned long long> smem_set{0}, carve_set{0};
        st = set_max_dynamic_smem(smem_set, fnp, (int)sizeof(SelSeqBwdSmem<CH>));
        if (st) return st;
        st = set_smem_carveout_max(carve_set, fnp);
        if (st) return st;
        sel_bwd_seq_kernel<CH><<<grid, CH * 8, sizeof(SelSeqBwdSmem<CH>), s>>>(
            reinterpret_cast<const bf16 *>(x), delta, A, reinterpret_cast<const bf16 *>(Bm),
            reinterpret_cast<const bf16 *>(Cm), ckpt, dy, dhT, dx, ddelta, dh0, w.partB, w.partC, w.partA, sg);
        st = check_launch(fn);
        if (st) return st;
        sel_reduce_bc_kernel<<<(unsigned int)((rows * kN + 255) / 256), 256, 0, s>>>(w.partB, w.partC, dB, dC, rows,
                                                                                    (int)(D / CH));
        st = check_launch(fn);
        if (st) return st;
        if (dA) {
            sel_reduce_a_kernel<<<(unsigned int)((D * kN + 31) / 32), kRedAWarps * 32, 0, s>>>(w.partA, dA, (int)B, 1,
                                                                                             (int)D);
            st = check_launch(fn);
        }
        return st;
    }
    static std::atomic<unsigned long long> smem_set{0};
    st = set_max_dynamic_smem(smem_set, reinterpret_cast<const void *>(sel_bwd_kernel), (int)sizeof(SelBwdSmem));
    if (st) return st;
    const unsigned int grid = (unsigned int)((size_t)p.gb.n_chunks * B * p.gb.n_cblk);
    sel_bwd_kernel<<<grid, kBwdThreads, sizeof(SelBwdSmem), s>>>(
        reinterpret_cast<const bf16 *>(x), delta, A, reinterpret_cast<const bf16 *>(Bm),
        reinterpret_cast<const bf16 *>(Cm), ckpt, dy, dhT, dx, ddelta, dh0, p.gb, w);
    st = check_launch(fn);
    if (st) return st;
    sel_reduce_bc_kernel<<<(unsigned int)((rows * kN + 255) / 256), 256, 0, s>>>(w.partB, w.partC, dB, dC, rows,
                                                                                p.gb.n_cblk);
    st = check_launch(fn);
    if (st) return st;
    if (dA) {
        sel_reduce_a_kernel<<<(unsigned int)((D * kN + 31) / 32), kRedAWarps * 32, 0, s>>>(w.partA, dA, (int)B,
                                                                                         p.g.n_chunks, (int)D);
        st = check_launch(fn);
    }
    return st;
}
