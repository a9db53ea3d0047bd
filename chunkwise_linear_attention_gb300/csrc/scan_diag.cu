// scan_diag.cu -- diagonal (vector-state) linear-recurrence scan, forward and
// backward, for GB300 (sm_103a).
//
// "Parallel Scan" (zerotofrontier.app), "The scan for one number of state",
// "A vectorized scan for diagonal states", "The backward pass is a scan in
// reverse"; "Parallel Scan" (aiwiki), the tiling remark: load a chunk, scan
// it on chip, carry one composed pair across the chunk boundary, never write
// intermediate states.
//
// Work decomposition (one warp = one chunk tile of TC = 8*L steps x 16
// channels):
//   lane = (sub, cg): cg in 0..3 picks 4 adjacent channels (one float4),
//   sub in 0..7 picks a run of L consecutive steps.  A warp load instruction
//   touches 8 rows x 64 contiguous bytes; the 4 warps of a block cover 64
//   adjacent channels (two whole 128-byte lines per row), so every line is
//   consumed by one block.
// Per tile:
//   1. every lane loads its L rows of (a, b) into registers (16-byte loads);
//   2. composes them sequentially into one pair (A, B) per channel;
//   3. warp-shuffle Hillis-Steele over the 8 runs (3 rounds) gives each run's
//      inclusive and exclusive prefix inside the chunk;
//   4. the last run's lanes publish the chunk aggregate, then walk back over
//      earlier chunks' published pairs (decoupled look-back) to obtain the
//      state entering the chunk, and publish the inclusive state;
//   5. every lane re-runs its L steps from its true starting state and
//      writes h once.
// HBM traffic is the algorithmic 12 B per element forward (read a, b; write
// h) and 20 B backward (read a, h, dh; write da, db), plus 12 B of look-back
// payload per chunk and channel (about 0.2 B per element, L2-resident).
#include "cla_internal.cuh"

namespace cla {
namespace {

constexpr int kSub = 8;      // runs per chunk (lanes along time)
constexpr int kCg = 4;       // lanes along channels
constexpr int kWarps = 4;    // warps per block (4 blocks per SM forward, 3 backward: measured best)
constexpr int kL = 8;        // steps per run
constexpr int kTc = kSub * kL;  // steps per chunk

template <int VEC>
struct VecIO;

template <>
struct VecIO<4> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[4]) {
        float4 x = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    static __device__ __forceinline__ void load_cs(const float *p, float (&v)[4]) {
        float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&v)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(v[0], v[1], v[2], v[3]));
    }
};

template <>
struct VecIO<1> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[1]) { v[0] = __ldg(p); }
    static __device__ __forceinline__ void load_cs(const float *p, float (&v)[1]) { v[0] = __ldcs(p); }
    static __device__ __forceinline__ void store(float *p, const float (&v)[1]) { __stcs(p, v[0]); }
};

// Look-back payload: per (chunk, batch row, warp column, channel group) and
// per channel, three 32-bit words -- the chunk's decay product A, its
// composed input B, and the state at its far edge (inclusive).  A word is 0
// until it is written (the launch clears them) and a written word is never 0:
// a value of +0.0f is stored as -0.0f, which every later use treats alike
// (a * (-0) + b and a * (+0) + b differ at most in the sign of a zero sum).
// A word is written and read with one relaxed 32-bit access, which is
// single-copy atomic, so a reader that sees a nonzero word sees the value: no
// memory fence is on the critical path.  (Each element of the 16-byte vector
// accesses below is such an access.)
struct ScanWs {
    WsHeader *hdr;
    unsigned int *words;  // [unit][3][4]
};

constexpr unsigned int kWordA = 0, kWordB = 1, kWordIncl = 2;

__device__ __forceinline__ unsigned int pub_bits(float v) {
    const unsigned int b = __float_as_uint(v);
    return b != 0u ? b : 0x80000000u;
}

template <int VEC>
__device__ __forceinline__ void publish(const ScanWs &ws, size_t u, unsigned int kind, const float (&v)[VEC]) {
    unsigned int *p = ws.words + (u * 3 + kind) * 4;
    if constexpr (VEC == 4)
        asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(pub_bits(v[0])),
                     "r"(pub_bits(v[1])), "r"(pub_bits(v[2])), "r"(pub_bits(v[3]))
                     : "memory");
    else
        asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(pub_bits(v[0])) : "memory");
}

template <int VEC>
__device__ __forceinline__ bool peek_words(const unsigned int *p, unsigned int (&w)[VEC]) {
    if constexpr (VEC == 4)
        asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "l"(p)
                     : "memory");
    else
        asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(w[0]) : "l"(p) : "memory");
    bool all = true;
#pragma unroll
    for (int i = 0; i < VEC; ++i) all = all && w[i] != 0u;
    return all;
}

// One step of the look-back walk at unit `up`: returns 2 when the unit's
// inclusive state was found (res = accA * incl + accB), 1 when its aggregate
// was composed into (accA, accB), 0 when the bounded wait gave up.
template <int VEC>
__device__ __forceinline__ unsigned int look_at(const ScanWs &ws, size_t up, float (&accA)[VEC], float (&accB)[VEC],
                                                float (&res)[VEC], unsigned int where) {
    const unsigned int *base = ws.words + up * 12;
    for (unsigned int it = 0; it < kSpinLimit; ++it) {
        unsigned int wi[VEC];
        if (peek_words<VEC>(base + kWordIncl * 4, wi)) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) res[i] = fmaf(accA[i], __uint_as_float(wi[i]), accB[i]);
            return 2u;
        }
        unsigned int wa[VEC], wb[VEC];
        const bool ra = peek_words<VEC>(base + kWordA * 4, wa);
        const bool rb = peek_words<VEC>(base + kWordB * 4, wb);
        if (ra && rb) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) {  // the unit's chunk happened before acc
                accB[i] = fmaf(accA[i], __uint_as_float(wb[i]), accB[i]);
                accA[i] *= __uint_as_float(wa[i]);
            }
            return 1u;
        }
        if (it >= 8) __nanosleep(100);
    }
    atomicOr(&ws.hdr->error, kErrTimeout);
    atomicExch(&ws.hdr->where, where);
    return 0u;
}

struct ScanGeom {
    int B, D, n_chunks, n_cw, n_cblk;
    long long T;
};

__host__ __device__ inline size_t scan_units(const ScanGeom &g) {
    return (size_t)g.n_chunks * g.B * g.n_cw * kCg;
}

__device__ __forceinline__ size_t unit_index(const ScanGeom &g, int chunk, int b, int cw, int cg) {
    return (((size_t)chunk * g.B + b) * g.n_cw + cw) * kCg + cg;
}

// ------------------------------------------------------------------ forward
// BLELLOCH selects how the 8 runs of a chunk are composed: Hillis-Steele
// (3 rounds, every run combines) or a Blelloch up-sweep / down-sweep (6 rounds,
// fewer combines), the latter kept as a measured alternative.
// STATES: instead of h, write only the state entering every chunk,
// h_in[chunk][B][D] (the backward's recompute path rebuilds h from it).
template <int VEC, bool BLELLOCH = false, bool STATES = false>
__global__ void __launch_bounds__(kWarps * 32, 4)
scan_diag_fwd_kernel(const float *__restrict__ a, const float *__restrict__ b,
                     const float *__restrict__ h0, float *__restrict__ h,
                     float *__restrict__ hT, ScanGeom g, ScanWs ws) {
    __shared__ unsigned int s_ticket;
    if (threadIdx.x == 0) s_ticket = atomicAdd(&ws.hdr->ticket[0], 1u);
    __syncthreads();
    const unsigned int tk = s_ticket;
    const int per_chunk = g.B * g.n_cblk;
    const int chunk = (int)(tk / per_chunk);
    const int rem = (int)(tk % per_chunk);
    const int bi = rem / g.n_cblk;
    const int cw = (rem % g.n_cblk) * kWarps + (threadIdx.x >> 5);
    if (cw >= g.n_cw) return;  // whole warp idle: nobody waits on it
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 2, cg = lane & 3;
    const int c0 = cw * (kCg * VEC) + cg * VEC;
    const bool cok = c0 < g.D;
    const long long t_begin = (long long)chunk * kTc + sub * kL;

    float av[kL][VEC], bv[kL][VEC];
#pragma unroll
    for (int i = 0; i < kL; ++i) {
        const long long t = t_begin + i;
        if (cok && t < g.T) {
            const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
            VecIO<VEC>::load_cs(a + idx, av[i]);
            VecIO<VEC>::load_cs(b + idx, bv[i]);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) { av[i][v] = 1.f; bv[i][v] = 0.f; }
        }
    }
    // 2. sequential composition of this lane's run
    float A[VEC], Bc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bc[v] = 0.f; }
#pragma unroll
    for (int i = 0; i < kL; ++i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Bc[v] = fmaf(av[i][v], Bc[v], bv[i][v]);
            A[v] *= av[i][v];
        }
    float Aex[VEC], Bex[VEC];  // prefix of the runs before this one
    if constexpr (!BLELLOCH) {
        // 3. Hillis-Steele across the 8 runs: combine with the run 1, 2, 4 to the left.
#pragma unroll
        for (int off = 1; off < kSub; off <<= 1) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float pa = __shfl_up_sync(0xffffffffu, A[v], off * kCg);
                const float pb = __shfl_up_sync(0xffffffffu, Bc[v], off * kCg);
                if (sub >= off) {  // (pa, pb) happened first
                    Bc[v] = fmaf(A[v], pb, Bc[v]);
                    A[v] *= pa;
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Aex[v] = __shfl_up_sync(0xffffffffu, A[v], kCg);
            Bex[v] = __shfl_up_sync(0xffffffffu, Bc[v], kCg);
            if (sub == 0) { Aex[v] = 1.f; Bex[v] = 0.f; }
        }
    } else {
        // 3'. Blelloch: up-sweep (run s with (s + 1) % 2st == 0 folds in run s - st, which
        // happened first); the last run then holds the chunk's pair.
#pragma unroll
        for (int st = 1; st < kSub; st <<= 1) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float pa = __shfl_up_sync(0xffffffffu, A[v], st * kCg);
                const float pb = __shfl_up_sync(0xffffffffu, Bc[v], st * kCg);
                if (((sub + 1) & (2 * st - 1)) == 0) {
                    Bc[v] = fmaf(A[v], pb, Bc[v]);
                    A[v] *= pa;
                }
            }
        }
        // down-sweep from the identity at the last run: a right node becomes (its prefix, then
        // the left subtree), a left node takes the right node's prefix.
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Aex[v] = (sub == kSub - 1) ? 1.f : A[v];
            Bex[v] = (sub == kSub - 1) ? 0.f : Bc[v];
        }
#pragma unroll
        for (int st = kSub / 2; st >= 1; st >>= 1) {
            const bool right = ((sub + 1) & (2 * st - 1)) == 0;
            const bool left = ((sub + 1 + st) & (2 * st - 1)) == 0;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float la = __shfl_up_sync(0xffffffffu, Aex[v], st * kCg);
                const float lb = __shfl_up_sync(0xffffffffu, Bex[v], st * kCg);
                const float ra = __shfl_down_sync(0xffffffffu, Aex[v], st * kCg);
                const float rb = __shfl_down_sync(0xffffffffu, Bex[v], st * kCg);
                if (right) {
                    Bex[v] = fmaf(la, Bex[v], lb);
                    Aex[v] *= la;
                } else if (left) {
                    Aex[v] = ra;
                    Bex[v] = rb;
                }
            }
        }
    }
    // 4. decoupled look-back by the lanes holding the chunk aggregate
    float carry[VEC];
    if (sub == kSub - 1) {
        const size_t u = unit_index(g, chunk, bi, cw, cg);
        float hin[VEC];
        if (chunk == 0) {
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                hin[v] = (h0 != nullptr && cok) ? h0[(size_t)bi * g.D + c0 + v] : 0.f;
        } else {
            publish<VEC>(ws, u, kWordA, A);
            publish<VEC>(ws, u, kWordB, Bc);
            float accA[VEC], accB[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) { accA[v] = 1.f; accB[v] = 0.f; hin[v] = 0.f; }
            for (int j = chunk - 1;; --j) {
                const unsigned int f = look_at<VEC>(ws, unit_index(g, j, bi, cw, cg), accA, accB, hin, 1u);
                if (f != 1u) break;  // inclusive found (or the wait gave up)
                if (j == 0) {        // reached the sequence start: apply h0
#pragma unroll
                    for (int v = 0; v < VEC; ++v) {
                        const float s0 = (h0 != nullptr && cok) ? h0[(size_t)bi * g.D + c0 + v] : 0.f;
                        hin[v] = fmaf(accA[v], s0, accB[v]);
                    }
                    break;
                }
            }
        }
        float inc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { inc[v] = fmaf(A[v], hin[v], Bc[v]); carry[v] = hin[v]; }
        publish<VEC>(ws, u, kWordIncl, inc);
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) carry[v] = __shfl_sync(0xffffffffu, carry[v], (kSub - 1) * kCg + cg);
    if constexpr (STATES) {
        if (sub == 0 && cok) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) h[((size_t)chunk * g.B + bi) * g.D + c0 + v] = carry[v];
        }
        if (hT == nullptr) return;
    }
    // 5. re-run this lane's steps from its true starting state; write h once
    float hs[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) hs[v] = fmaf(Aex[v], carry[v], Bex[v]);
#pragma unroll
    for (int i = 0; i < kL; ++i) {
        const long long t = t_begin + i;
#pragma unroll
        for (int v = 0; v < VEC; ++v) hs[v] = fmaf(av[i][v], hs[v], bv[i][v]);
        if (cok && t < g.T) {
            const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
            if constexpr (!STATES) VecIO<VEC>::store(h + idx, hs);
            if (hT != nullptr && t == g.T - 1)
#pragma unroll
                for (int v = 0; v < VEC; ++v) hT[(size_t)bi * g.D + c0 + v] = hs[v];
        }
    }
}

// ------------------------------------------------------------------ backward
// Reversed time: hbar_t = a'_t hbar_{t+1} + g_t with a'_t = a_{t+1}
// (a'_{T-1} = 1 and g_{T-1} includes dhT), i.e. the forward scan on reversed
// arrays with the decays shifted by one place.
//
// RECOMP: h is not given.  `h` then points at the state entering every chunk,
// h_in[chunk][B][D] (written by the STATES forward), and `b` at the forward's
// inputs; each lane rebuilds h_{t-1} over its run from them -- the run's own
// (a, b) composed forward, Hillis-Steele across the runs of the chunk, applied
// to the chunk's entry state -- instead of reading it ("The backward pass is a
// scan in reverse": store the states or recompute them).
template <int VEC, bool RECOMP = false>
__global__ void __launch_bounds__(kWarps * 32, 3)
scan_diag_bwd_kernel(const float *__restrict__ a, const float *__restrict__ b,
                     const float *__restrict__ h0,
                     const float *__restrict__ h, const float *__restrict__ dh,
                     const float *__restrict__ dhT, float *__restrict__ da,
                     float *__restrict__ db, float *__restrict__ dh0, ScanGeom g,
                     ScanWs ws) {
    __shared__ unsigned int s_ticket;
    if (threadIdx.x == 0) s_ticket = atomicAdd(&ws.hdr->ticket[1], 1u);
    __syncthreads();
    const unsigned int tk = s_ticket;
    const int per_chunk = g.B * g.n_cblk;
    const int chunk = g.n_chunks - 1 - (int)(tk / per_chunk);
    const int rem = (int)(tk % per_chunk);
    const int bi = rem / g.n_cblk;
    const int cw = (rem % g.n_cblk) * kWarps + (threadIdx.x >> 5);
    if (cw >= g.n_cw) return;
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 2, cg = lane & 3;
    const int c0 = cw * (kCg * VEC) + cg * VEC;
    const bool cok = c0 < g.D;
    const long long t_begin = (long long)chunk * kTc + sub * kL;

    // h_{t-1} is only needed in the last pass: stage it in shared memory now
    // (asynchronously, holding no registers) so its latency overlaps the rest.
    __shared__ __align__(16) float s_hp[RECOMP ? 1 : kL][kWarps * 32][VEC];
    if constexpr (!RECOMP) {
#pragma unroll
        for (int i = 0; i < kL; ++i) {
            const long long t = t_begin + i;
            const bool ok = cok && t >= 1 && t < g.T;
            const float *src = h + (ok ? ((size_t)bi * g.T + t - 1) * g.D + c0 : 0);
            const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&s_hp[i][threadIdx.x][0]));
            if (VEC == 4)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                             "r"(ok ? 16u : 0u)
                             : "memory");
            else
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 4u : 0u)
                             : "memory");
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    }
    // RECOMP: the forward inputs b_t of this run and a_t of its first step (a_t of the
    // others is ap[i - 1] below); hp[i] becomes h_{t-1}
    float hp[RECOMP ? kL : 1][VEC], a_first[VEC];
    if constexpr (RECOMP) {
#pragma unroll
        for (int i = 0; i < kL; ++i) {
            const long long t = t_begin + i;
            if (cok && t < g.T) {
                VecIO<VEC>::load_cs(b + ((size_t)bi * g.T + t) * g.D + c0, hp[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) hp[i][v] = 0.f;
            }
        }
        if (cok && t_begin < g.T) {
            VecIO<VEC>::load(a + ((size_t)bi * g.T + t_begin) * g.D + c0, a_first);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) a_first[v] = 1.f;
        }
    }
    float ap[kL][VEC], gv[kL][VEC];
#pragma unroll
    for (int i = 0; i < kL; ++i) {
        const long long t = t_begin + i;
        if (cok && t < g.T) {
            const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
            VecIO<VEC>::load_cs(dh + idx, gv[i]);
            if (t + 1 < g.T) {
                VecIO<VEC>::load(a + idx + g.D, ap[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    ap[i][v] = 1.f;
                    if (dhT != nullptr) gv[i][v] += dhT[(size_t)bi * g.D + c0 + v];
                }
            }
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) { ap[i][v] = 1.f; gv[i][v] = 0.f; }
        }
    }
    // compose this lane's run from its last step down to its first
    float A[VEC], Bc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bc[v] = 0.f; }
#pragma unroll
    for (int i = kL - 1; i >= 0; --i)
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Bc[v] = fmaf(ap[i][v], Bc[v], gv[i][v]);
            A[v] *= ap[i][v];
        }
    // Hillis-Steele over the runs toward the chunk's start (suffix direction)
#pragma unroll
    for (int off = 1; off < kSub; off <<= 1) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float pa = __shfl_down_sync(0xffffffffu, A[v], off * kCg);
            const float pb = __shfl_down_sync(0xffffffffu, Bc[v], off * kCg);
            if (sub + off < kSub) {  // the later run (pa, pb) applies first
                Bc[v] = fmaf(A[v], pb, Bc[v]);
                A[v] *= pa;
            }
        }
    }
    float Aex[VEC], Bex[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        Aex[v] = __shfl_down_sync(0xffffffffu, A[v], kCg);
        Bex[v] = __shfl_down_sync(0xffffffffu, Bc[v], kCg);
        if (sub == kSub - 1) { Aex[v] = 1.f; Bex[v] = 0.f; }
    }
    if constexpr (RECOMP) {
        // forward composition of this run, then Hillis-Steele across the runs of the chunk
        // (exclusive prefix), applied to the chunk's entry state: h entering this run
        float FA[VEC], FB[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { FA[v] = 1.f; FB[v] = 0.f; }
#pragma unroll
        for (int i = 0; i < kL; ++i)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float at = i == 0 ? a_first[v] : ap[i - 1][v];
                FB[v] = fmaf(at, FB[v], hp[i][v]);
                FA[v] *= at;
            }
#pragma unroll
        for (int off = 1; off < kSub; off <<= 1) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float pa = __shfl_up_sync(0xffffffffu, FA[v], off * kCg);
                const float pb = __shfl_up_sync(0xffffffffu, FB[v], off * kCg);
                if (sub >= off) {
                    FB[v] = fmaf(FA[v], pb, FB[v]);
                    FA[v] *= pa;
                }
            }
        }
        float hs[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            float ea = __shfl_up_sync(0xffffffffu, FA[v], kCg);
            float eb = __shfl_up_sync(0xffffffffu, FB[v], kCg);
            if (sub == 0) { ea = 1.f; eb = 0.f; }
            const float s0 = cok ? __ldcg(h + ((size_t)chunk * g.B + bi) * g.D + c0 + v) : 0.f;
            hs[v] = fmaf(ea, s0, eb);
        }
#pragma unroll
        for (int i = 0; i < kL; ++i)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float at = i == 0 ? a_first[v] : ap[i - 1][v];
                const float bt = hp[i][v];
                hp[i][v] = hs[v];
                hs[v] = fmaf(at, hs[v], bt);
            }
    }
    float carry[VEC];
    if (sub == 0) {
        const size_t u = unit_index(g, chunk, bi, cw, cg);
        float hin[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) hin[v] = 0.f;
        if (chunk != g.n_chunks - 1) {
            publish<VEC>(ws, u, kWordA, A);
            publish<VEC>(ws, u, kWordB, Bc);
            float accA[VEC], accB[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) { accA[v] = 1.f; accB[v] = 0.f; }
            for (int j = chunk + 1;; ++j) {
                const unsigned int f = look_at<VEC>(ws, unit_index(g, j, bi, cw, cg), accA, accB, hin, 2u);
                if (f != 1u) break;
                if (j == g.n_chunks - 1) {  // past the sequence end: nothing more flows in
#pragma unroll
                    for (int v = 0; v < VEC; ++v) hin[v] = accB[v];
                    break;
                }
            }
        }
        float inc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { inc[v] = fmaf(A[v], hin[v], Bc[v]); carry[v] = hin[v]; }
        publish<VEC>(ws, u, kWordIncl, inc);
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) carry[v] = __shfl_sync(0xffffffffu, carry[v], cg);
    if constexpr (!RECOMP) asm volatile("cp.async.wait_group 0;\n" ::: "memory");  // own copies of h_{t-1}
    float hb[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) hb[v] = fmaf(Aex[v], carry[v], Bex[v]);
#pragma unroll
    for (int i = kL - 1; i >= 0; --i) {
        const long long t = t_begin + i;
#pragma unroll
        for (int v = 0; v < VEC; ++v) hb[v] = fmaf(ap[i][v], hb[v], gv[i][v]);
        if (cok && t < g.T) {
            const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
            float hprev[VEC];  // h_{t-1}
            if constexpr (RECOMP) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) hprev[v] = hp[i][v];
            } else if (t >= 1) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) hprev[v] = s_hp[i][threadIdx.x][v];
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) hprev[v] = (h0 != nullptr) ? h0[(size_t)bi * g.D + c0 + v] : 0.f;
            }
            float dav[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) dav[v] = hb[v] * hprev[v];
            VecIO<VEC>::store(db + idx, hb);
            VecIO<VEC>::store(da + idx, dav);
            if (dh0 != nullptr && t == 0) {
                float a1[VEC];
                VecIO<VEC>::load(a + idx, a1);
#pragma unroll
                for (int v = 0; v < VEC; ++v) dh0[(size_t)bi * g.D + c0 + v] = a1[v] * hb[v];
            }
        }
    }
}

// ------------------------------------------------------------------ short sequences
// A problem too small to fill the GPU with chunk blocks (at most kSmallBlocks
// channel groups, each at most kSmallMaxChunks chunks long) runs in one block
// per (batch row, channel group), with no workspace and no cross-block
// look-back (it only clears the workspace header's status): warp w owns a
// contiguous run of chunks; it folds them into one
// pair per channel (phase 1), the block composes the warps' pairs in shared
// memory onto h0, and each warp re-runs its chunks from its true incoming
// state and writes h (phase 2; the re-read hits L2).  Inside a chunk the
// composition is the one of scan_diag_fwd_kernel: a sequential run per lane,
// then Hillis-Steele across the 8 runs.
constexpr int kSmallWarps = 16;        // one chunk per warp up to 1024 steps
constexpr int kSmallMaxChunks = 64;
constexpr long long kSmallBlocks = 152;

template <int VEC>
__global__ void __launch_bounds__(kSmallWarps * 32)
scan_diag_fwd_small_kernel(const float *__restrict__ a, const float *__restrict__ b,
                           const float *__restrict__ h0, float *__restrict__ h,
                           float *__restrict__ hT, ScanGeom g, WsHeader *hdr) {
    __shared__ float sA[kSmallWarps][kCg * VEC], sB[kSmallWarps][kCg * VEC];
    // this call's status, for cla_check_status: the kernel has no cross-block wait to give up
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        hdr->error = 0u;
        hdr->where = 0u;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane >> 2, cg = lane & 3;
    const int bi = blockIdx.y, cw = blockIdx.x;
    const int c0 = cw * (kCg * VEC) + cg * VEC;
    const bool cok = c0 < g.D;
    const int per = (g.n_chunks + kSmallWarps - 1) / kSmallWarps;
    const int ch_begin = min(warp * per, g.n_chunks), ch_end = min(ch_begin + per, g.n_chunks);

    // the runs of one chunk: this lane's steps, its run's pair and its prefix within the chunk,
    // and the chunk's pair (the last run's inclusive prefix, on every lane)
    float av[kL][VEC], bv[kL][VEC], Aex[VEC], Bex[VEC], CA[VEC], CB[VEC];
    auto chunk_pairs = [&](int chunk) {
        const long long t_begin = (long long)chunk * kTc + sub * kL;
#pragma unroll
        for (int i = 0; i < kL; ++i) {
            const long long t = t_begin + i;
            if (cok && t < g.T) {
                const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
                VecIO<VEC>::load(a + idx, av[i]);
                VecIO<VEC>::load(b + idx, bv[i]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) { av[i][v] = 1.f; bv[i][v] = 0.f; }
            }
        }
        float A[VEC], Bc[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) { A[v] = 1.f; Bc[v] = 0.f; }
#pragma unroll
        for (int i = 0; i < kL; ++i)
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                Bc[v] = fmaf(av[i][v], Bc[v], bv[i][v]);
                A[v] *= av[i][v];
            }
#pragma unroll
        for (int off = 1; off < kSub; off <<= 1) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float pa = __shfl_up_sync(0xffffffffu, A[v], off * kCg);
                const float pb = __shfl_up_sync(0xffffffffu, Bc[v], off * kCg);
                if (sub >= off) {
                    Bc[v] = fmaf(A[v], pb, Bc[v]);
                    A[v] *= pa;
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            Aex[v] = __shfl_up_sync(0xffffffffu, A[v], kCg);
            Bex[v] = __shfl_up_sync(0xffffffffu, Bc[v], kCg);
            if (sub == 0) { Aex[v] = 1.f; Bex[v] = 0.f; }
            CA[v] = __shfl_sync(0xffffffffu, A[v], (kSub - 1) * kCg + cg);
            CB[v] = __shfl_sync(0xffffffffu, Bc[v], (kSub - 1) * kCg + cg);
        }
    };

    // phase 1: this warp's chunks folded into one pair per channel
    float SA[VEC], SB[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) { SA[v] = 1.f; SB[v] = 0.f; }
    for (int chunk = ch_begin; chunk < ch_end; ++chunk) {
        chunk_pairs(chunk);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            SB[v] = fmaf(CA[v], SB[v], CB[v]);
            SA[v] *= CA[v];
        }
    }
    if (sub == 0) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            sA[warp][cg * VEC + v] = SA[v];
            sB[warp][cg * VEC + v] = SB[v];
        }
    }
    __syncthreads();
    // the state entering this warp's chunks: h0, then the earlier warps' pairs in order
    float carry[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) carry[v] = (h0 != nullptr && cok) ? h0[(size_t)bi * g.D + c0 + v] : 0.f;
    for (int w = 0; w < warp; ++w)
#pragma unroll
        for (int v = 0; v < VEC; ++v) carry[v] = fmaf(sA[w][cg * VEC + v], carry[v], sB[w][cg * VEC + v]);

    // phase 2: re-run from the true state, write h once
    const bool one = (ch_end - ch_begin) == 1;  // the registers still hold the chunk's steps and pairs
    for (int chunk = ch_begin; chunk < ch_end; ++chunk) {
        if (!one) chunk_pairs(chunk);
        const long long t_begin = (long long)chunk * kTc + sub * kL;
        float hs[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) hs[v] = fmaf(Aex[v], carry[v], Bex[v]);
#pragma unroll
        for (int i = 0; i < kL; ++i) {
            const long long t = t_begin + i;
#pragma unroll
            for (int v = 0; v < VEC; ++v) hs[v] = fmaf(av[i][v], hs[v], bv[i][v]);
            if (cok && t < g.T) {
                const size_t idx = ((size_t)bi * g.T + t) * g.D + c0;
                VecIO<VEC>::store(h + idx, hs);
                if (hT != nullptr && t == g.T - 1)
#pragma unroll
                    for (int v = 0; v < VEC; ++v) hT[(size_t)bi * g.D + c0 + v] = hs[v];
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) carry[v] = fmaf(CA[v], carry[v], CB[v]);
    }
}

// ------------------------------------------------------------------ host side
struct Plan {
    ScanGeom g;
    int vec;
    size_t words_off, total;
    // the backward's recompute path also keeps the state entering every chunk,
    // [n_chunks][B][D] fp32, after the look-back words
    size_t states_off, total_recomp;
};

Plan make_plan(int64_t B, int64_t T, int64_t D, int vec) {
    Plan p;
    p.vec = vec;
    p.g.B = (int)B;
    p.g.D = (int)D;
    p.g.T = T;
    p.g.n_chunks = (int)((T + kTc - 1) / kTc);
    const int per_warp = kCg * vec;
    p.g.n_cw = (int)((D + per_warp - 1) / per_warp);
    p.g.n_cblk = (p.g.n_cw + kWarps - 1) / kWarps;
    p.words_off = sizeof(WsHeader);
    p.total = p.words_off + scan_units(p.g) * 12 * sizeof(unsigned int);
    p.states_off = align_up(p.total, 256);
    p.total_recomp = p.states_off + (size_t)p.g.n_chunks * (size_t)B * (size_t)D * sizeof(float);
    return p;
}

ScanWs bind_ws(const Plan &p, void *ws) {
    char *base = static_cast<char *>(ws);
    ScanWs w;
    w.hdr = reinterpret_cast<WsHeader *>(base);
    w.words = reinterpret_cast<unsigned int *>(base + p.words_off);
    return w;
}

// Sizes every kernel and plan of this file handles (non-negative sizes): the
// grid stays below 2^31 blocks and every count fits its integer type.
bool sizes_fit(int64_t B, int64_t T, int64_t D) {
    if (D > (1ll << 30) || B > (1ll << 24) || T > (1ll << 40)) return false;
    const int64_t n_chunks = (T + kTc - 1) / kTc;
    const int64_t n_cblk = ((D + 15) / 16 + kWarps - 1) / kWarps;
    return product_below({n_chunks, B, (D + 3) / 4 + kWarps - 1}, 2147483648.0) &&
           product_below({n_chunks, B, n_cblk}, 2147483648.0);
}

int check_sizes(const char *fn, int64_t B, int64_t T, int64_t D) {
    if (B < 0 || T < 0 || D < 0) return fail(CLA_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!sizes_fit(B, T, D)) return fail(CLA_ERR_UNSUPPORTED, "%s: size out of range for one launch", fn);
    return CLA_OK;
}

}  // namespace
}  // namespace cla

using namespace cla;

extern "C" size_t cla_scan_diag_workspace_size(int64_t B, int64_t T, int64_t D) {
    if (B < 0 || T < 0 || D < 0 || !sizes_fit(B, T, D)) return 0;
    // the scalar-channel layout needs the most units; size for it
    const Plan p1 = make_plan(B, T, D, 1);
    const Plan p4 = make_plan(B, T, D, 4);
    return p1.total_recomp > p4.total_recomp ? p1.total_recomp : p4.total_recomp;
}

extern "C" size_t cla_scan_diag_workspace(int64_t B, int64_t T, int64_t D) {
    return cla_scan_diag_workspace_size(B, T, D);
}

namespace {
int scan_fwd(const char *fn, bool blelloch, const float *a, const float *b, const float *h0, float *h, float *hT,
             int64_t B, int64_t T, int64_t D, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    int st = check_sizes(fn, B, T, D);
    if (st) return st;
    if (!aligned_or_null({a, b, h0, h, hT}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: fp32 tensors must be 4-byte aligned", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return CLA_OK;
    if (T == 0) {
        if (hT) {
            if (h0) CLA_CUDA_TRY(cudaMemcpyAsync(hT, h0, sizeof(float) * B * D, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(hT, 0, sizeof(float) * B * D, s), fn);
        }
        return CLA_OK;
    }
    if (!a || !b || !h) return fail(CLA_ERR_INVALID_ARG, "%s: a, b and h are required", fn);
    if (!ws) return fail(CLA_ERR_WORKSPACE, "%s: workspace is NULL", fn);
    if (!aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace not 16-byte aligned", fn);
    const bool v4 = (D % 4 == 0) && aligned16(a) && aligned16(b) && aligned16(h);
    const Plan p = make_plan(B, T, D, v4 ? 4 : 1);
    if (ws_bytes < p.total) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, p.total);
    if (!blelloch && p.g.n_chunks <= kSmallMaxChunks && (long long)p.g.B * p.g.n_cw <= kSmallBlocks) {
        // short sequence, few channel groups: one block per group, no workspace traffic; one
        // channel per lane while that still fits one block per SM (more blocks: more loads in
        // flight at once, the call being bound by their latency)
        WsHeader *hdr = static_cast<WsHeader *>(ws);
        const Plan p1 = make_plan(B, T, D, 1);
        if (!v4 || (long long)p1.g.B * p1.g.n_cw <= kSmallBlocks) {
            const dim3 grid((unsigned int)p1.g.n_cw, (unsigned int)p1.g.B);
            scan_diag_fwd_small_kernel<1><<<grid, kSmallWarps * 32, 0, s>>>(a, b, h0, h, hT, p1.g, hdr);
        } else {
            const dim3 grid((unsigned int)p.g.n_cw, (unsigned int)p.g.B);
            scan_diag_fwd_small_kernel<4><<<grid, kSmallWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, hdr);
        }
        return check_launch(fn);
    }
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.total, s), fn);
    const ScanWs w = bind_ws(p, ws);
    const unsigned int grid = (unsigned int)((size_t)p.g.n_chunks * p.g.B * p.g.n_cblk);
    if (blelloch) {
        if (v4) scan_diag_fwd_kernel<4, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
        else scan_diag_fwd_kernel<1, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
    } else {
        if (v4) scan_diag_fwd_kernel<4><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
        else scan_diag_fwd_kernel<1><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
    }
    return check_launch(fn);
}
}  // namespace

extern "C" int cla_scan_diag_fwd(const float *a, const float *b, const float *h0, float *h,
                                 float *hT, int64_t B, int64_t T, int64_t D, void *ws,
                                 size_t ws_bytes, void *stream) {
    return scan_fwd("cla_scan_diag_fwd", false, a, b, h0, h, hT, B, T, D, ws, ws_bytes, stream);
}

extern "C" int cla_scan_diag_fwd_blelloch(const float *a, const float *b, const float *h0, float *h,
                                          float *hT, int64_t B, int64_t T, int64_t D, void *ws,
                                          size_t ws_bytes, void *stream) {
    return scan_fwd("cla_scan_diag_fwd_blelloch", true, a, b, h0, h, hT, B, T, D, ws, ws_bytes, stream);
}

extern "C" int cla_scan_diag_bwd(const float *a, const float *b, const float *h0, const float *h,
                                 const float *dh, const float *dhT, float *da, float *db,
                                 float *dh0, int64_t B, int64_t T, int64_t D, void *ws,
                                 size_t ws_bytes, void *stream) {
    clear_error();
    const char *fn = "cla_scan_diag_bwd";
    int st = check_sizes(fn, B, T, D);
    if (st) return st;
    if (!aligned_or_null({a, b, h0, h, dh, dhT, da, db, dh0}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: fp32 tensors must be 4-byte aligned", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return CLA_OK;
    if (T == 0) {  // h_T = h0: the gradient passes straight through
        if (dh0) {
            if (dhT) CLA_CUDA_TRY(cudaMemcpyAsync(dh0, dhT, sizeof(float) * B * D, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(dh0, 0, sizeof(float) * B * D, s), fn);
        }
        return CLA_OK;
    }
    if (!a || !dh || !da || !db) return fail(CLA_ERR_INVALID_ARG, "%s: a, dh, da and db are required", fn);
    if (!h && !b) return fail(CLA_ERR_INVALID_ARG, "%s: give h (the forward's states) or b (to recompute them)", fn);
    if (!ws) return fail(CLA_ERR_WORKSPACE, "%s: workspace is NULL", fn);
    if (!aligned16(ws)) return fail(CLA_ERR_WORKSPACE, "%s: workspace not 16-byte aligned", fn);
    const bool recomp = (h == nullptr);
    const float *hsrc = recomp ? b : h;  // the tensor read in place of h
    const bool v4 = (D % 4 == 0) && aligned16(a) && aligned16(hsrc) && aligned16(dh) && aligned16(da) &&
                    aligned16(db);
    const Plan p = make_plan(B, T, D, v4 ? 4 : 1);
    const size_t need = recomp ? p.total_recomp : p.total;
    if (ws_bytes < need) return fail(CLA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, need);
    const ScanWs w = bind_ws(p, ws);
    const unsigned int grid = (unsigned int)((size_t)p.g.n_chunks * p.g.B * p.g.n_cblk);
    float *states = reinterpret_cast<float *>(static_cast<char *>(ws) + p.states_off);
    if (recomp) {
        // the state entering every chunk, by the forward scan without writing h
        CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.total, s), fn);
        if (v4) scan_diag_fwd_kernel<4, false, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, states, nullptr, p.g, w);
        else scan_diag_fwd_kernel<1, false, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, states, nullptr, p.g, w);
        st = check_launch(fn);
        if (st) return st;
    }
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.total, s), fn);
    if (recomp) {
        if (v4) scan_diag_bwd_kernel<4, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, states, dh, dhT, da, db, dh0, p.g, w);
        else scan_diag_bwd_kernel<1, true><<<grid, kWarps * 32, 0, s>>>(a, b, h0, states, dh, dhT, da, db, dh0, p.g, w);
    } else {
        if (v4) scan_diag_bwd_kernel<4><<<grid, kWarps * 32, 0, s>>>(a, nullptr, h0, h, dh, dhT, da, db, dh0, p.g, w);
        else scan_diag_bwd_kernel<1><<<grid, kWarps * 32, 0, s>>>(a, nullptr, h0, h, dh, dhT, da, db, dh0, p.g, w);
    }
    return check_launch(fn);
}

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot hand this library a workspace: a plugin inside a host
// framework that owns every device allocation and exposes no scratch space, a
// deployment whose device-memory footprint is fixed in advance, or a code
// path where an allocation call (its latency or its implicit synchronisation)
// is not allowed.  For them the forward diagonal scan can run with its
// look-back scratch in a statically sized device array that is part of the
// library image.  Each GPU that loads the library keeps this array for the
// life of the process.

namespace cla {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_scan_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array in the current device's context.  The name
// g_scan_noalloc_scratch is only a host-side stand-in in host code and must
// never be passed to a kernel directly.  The address is looked up on every
// call (the lookup allocates nothing): a cached address would go stale when
// the module is loaded again, after cudaDeviceReset or in another context.
int noalloc_scratch(const char *fn, void **out) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scan_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
        return fail(CLA_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", fn, cudaGetErrorString(e));
    *out = p;
    return CLA_OK;
}

}  // namespace
}  // namespace cla

extern "C" int cla_scan_diag_fwd_noalloc(const float *a, const float *b, const float *h0, float *h, float *hT,
                                         int64_t B, int64_t T, int64_t D, void *stream) {
    clear_error();
    const char *fn = "cla_scan_diag_fwd_noalloc";
    int st = check_sizes(fn, B, T, D);
    if (st) return st;
    if (!aligned_or_null({a, b, h0, h, hT}, 4))
        return fail(CLA_ERR_INVALID_ARG, "%s: fp32 tensors must be 4-byte aligned", fn);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return CLA_OK;
    if (T == 0) {
        if (hT) {
            if (h0) CLA_CUDA_TRY(cudaMemcpyAsync(hT, h0, sizeof(float) * B * D, cudaMemcpyDeviceToDevice, s), fn);
            else CLA_CUDA_TRY(cudaMemsetAsync(hT, 0, sizeof(float) * B * D, s), fn);
        }
        return CLA_OK;
    }
    if (!a || !b || !h) return fail(CLA_ERR_INVALID_ARG, "%s: a, b and h are required", fn);
    const bool v4 = (D % 4 == 0) && aligned16(a) && aligned16(b) && aligned16(h);
    const Plan p = make_plan(B, T, D, v4 ? 4 : 1);
    if (p.total > kNoAllocScratchBytes)
        return fail(CLA_ERR_UNSUPPORTED,
                    "%s: this size needs %zu bytes of scratch but the static array holds %zu; "
                    "use cla_scan_diag_fwd with a caller workspace",
                    fn, p.total, kNoAllocScratchBytes);
    void *ws = nullptr;
    st = noalloc_scratch(fn, &ws);
    if (st) return st;
    // tickets and flags must start at zero; the payload is always written before it is read
    CLA_CUDA_TRY(cudaMemsetAsync(ws, 0, p.total, s), fn);
    const ScanWs w = bind_ws(p, ws);
    const unsigned int grid = (unsigned int)((size_t)p.g.n_chunks * p.g.B * p.g.n_cblk);
    if (v4) scan_diag_fwd_kernel<4><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
    else scan_diag_fwd_kernel<1><<<grid, kWarps * 32, 0, s>>>(a, b, h0, h, hT, p.g, w);
    return check_launch(fn);
}

extern "C" int cla_scan_diag_noalloc_check_status(void *stream) {
    clear_error();
    const char *fn = "cla_scan_diag_noalloc_check_status";
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CLA_CUDA_TRY(cudaStreamSynchronize(s), fn);
    WsHeader hdr;
    // a copy into host memory: nothing is allocated
    CLA_CUDA_TRY(cudaMemcpyFromSymbol(&hdr, g_scan_noalloc_scratch, sizeof(hdr), 0, cudaMemcpyDeviceToHost), fn);
    if (hdr.error & kErrTimeout)
        return fail(CLA_ERR_TIMEOUT, "%s: a cross-block wait gave up (site %u)", fn, hdr.where);
    return CLA_OK;
}
