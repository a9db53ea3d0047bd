/*
 * cla.h -- C ABI of libcla.so: linear-recurrence scans and chunkwise decayed
 * linear attention, forward and backward, as hand-written CUDA for GB300
 * (sm_103a).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  Inputs are
 *    read, outputs are overwritten entirely; no pointer is retained after the
 *    call returns.  The library never allocates or frees device memory and
 *    never synchronises: it validates the arguments on the host, enqueues its
 *    kernels (and small memsets of its workspace) on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream) and returns.
 *  - Tensors are dense, row-major, with the innermost dimension last, and
 *    16-byte aligned.  `bf16` arguments are bfloat16 bit patterns (uint16_t).
 *    A pointer misaligned for the way a kernel reads or writes it (below its
 *    element size anywhere; below 16 bytes for the tensors loaded or stored
 *    in 16-byte pieces or by TMA) is rejected with CLA_ERR_INVALID_ARG
 *    before anything is enqueued.
 *  - Arguments marked [opt] may be NULL: an optional input then means zeros,
 *    an optional output is not written.
 *  - `ws`/`ws_bytes` is caller-owned scratch of at least the size returned by
 *    the matching *_workspace_size() query (16-byte aligned).  Its contents
 *    need not be initialised and are meaningless after the call.  Calls that
 *    may run concurrently must use distinct workspaces.
 *  - Errors: argument and shape errors are detected before anything is
 *    enqueued and return CLA_ERR_INVALID_ARG / CLA_ERR_UNSUPPORTED /
 *    CLA_ERR_WORKSPACE; a failed launch returns CLA_ERR_CUDA.  The kernels
 *    never trap: a cross-block wait that exceeds its iteration bound records
 *    a flag in the workspace and the block carries on; cla_check_status()
 *    reports it as CLA_ERR_TIMEOUT.  cla_last_error_message() gives a
 *    one-line description of the last failure on the calling host thread.
 *
 * Sources (page title and section):
 *   "Parallel Scan" (zerotofrontier.app/ssm/parallel-scan)
 *   "Lightning Attention-2" (arXiv 2401.04658, summary on paper-graph-ui)
 *   "Parallel Scan" (aiwiki.thehackersbrain.dev/entries/parallel-scan)
 */
#ifndef CLA_H_
#define CLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CLA_OK = 0,
    CLA_ERR_INVALID_ARG = 1, /* null required pointer, negative size, misalignment */
    CLA_ERR_UNSUPPORTED = 2, /* a size or head dimension this build has no kernel for */
    CLA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    CLA_ERR_TIMEOUT = 4,     /* a bounded cross-block wait gave up (see cla_check_status) */
    CLA_ERR_WORKSPACE = 5    /* ws is NULL, unaligned or smaller than required */
} cla_status;

/* Static, never-NULL name of a status code. */
const char *cla_status_string(int status);

/* Description of the last failing call on this host thread ("" if none). */
const char *cla_last_error_message(void);

/* Synchronises `stream`, then reports CLA_ERR_TIMEOUT if a kernel of the last
 * call that used `ws` gave up a cross-block wait, CLA_ERR_UNSUPPORTED if it
 * met data outside its range (cla_gla_fwd's decay bound), CLA_ERR_CUDA if the
 * stream holds an error, else CLA_OK.  `ws` must be the workspace of that
 * call. */
int cla_check_status(const void *ws, void *stream);
/* The same call under the name the boundary's plan gives it. */
int cla_check_device_status(const void *ws, void *stream);

/* Self-test of the failure path: launches one warp that polls a workspace
 * word nothing ever sets.  Its bounded wait gives up after about a second,
 * records the timeout in `ws` (16-byte aligned, at least 256 bytes: the
 * workspace header) and returns; a following
 * cla_check_status(ws, stream) then reports CLA_ERR_TIMEOUT.  No GPU fault,
 * trap or hang is involved. */
int cla_selftest_wait_timeout(void *ws, size_t ws_bytes, void *stream);

/* ======================================================================== */
/* Diagonal (vector-state) scan                                             */
/* ======================================================================== */

/* Bytes of workspace needed by cla_scan_diag_fwd / _bwd for [B, T, D]. */
size_t cla_scan_diag_workspace_size(int64_t B, int64_t T, int64_t D);
/* The same query under the name the boundary's plan gives it. */
size_t cla_scan_diag_workspace(int64_t B, int64_t T, int64_t D);

/* Forward: h_t = a_t * h_{t-1} + b_t elementwise over D channels, for
 * t = 1..T, from h_0 = h0 ("Parallel Scan", "The scan for one number of
 * state" and "A vectorized scan for diagonal states"; the initial state is
 * folded into the first step, "Scans over vector and matrix states").
 *   a, b   [B, T, D] fp32   decays and inputs
 *   h0     [B, D]    fp32   [opt] initial state (NULL = 0)
 *   h      [B, T, D] fp32   out: every state h_1..h_T
 *   hT     [B, D]    fp32   [opt] out: h_T (h0 when T = 0)
 * Each chunk of the sequence is composed inside one warp (a sequential run
 * per lane, then Hillis-Steele across lanes) and one composed (a, b) pair per
 * chunk and channel is carried across chunks by decoupled look-back; no
 * intermediate pair reaches HBM beyond that one per chunk. */
int cla_scan_diag_fwd(const float *a, const float *b, const float *h0, float *h,
                      float *hT, int64_t B, int64_t T, int64_t D, void *ws,
                      size_t ws_bytes, void *stream);

/* cla_scan_diag_fwd with the runs of a chunk composed by a Blelloch
 * up-sweep / down-sweep instead of Hillis-Steele ("Parallel Scan", the
 * work-efficient scan the page contrasts with Hillis-Steele; "Parallel Scan"
 * (aiwiki), the tree form).  Same arguments, layouts, workspace, ownership
 * and errors as cla_scan_diag_fwd, and the same results up to rounding order;
 * kept as a measured alternative (the up-sweep and down-sweep take six
 * shuffle rounds across the eight runs where Hillis-Steele takes three). */
int cla_scan_diag_fwd_blelloch(const float *a, const float *b, const float *h0,
                               float *h, float *hT, int64_t B, int64_t T,
                               int64_t D, void *ws, size_t ws_bytes, void *stream);

/* Backward ("Parallel Scan", "The backward pass is a scan in reverse"): with
 * direct gradients g_t = dh_t (plus dhT on h_T), the adjoint
 * hbar_t = g_t + a_{t+1} hbar_{t+1} is the same scan on reversed time with
 * the decays shifted by one; then db_t = hbar_t, da_t = hbar_t * h_{t-1},
 * dh0 = a_1 * hbar_1.  The states h_{t-1} are read from the forward's output
 * when `h` is given, else recomputed from (a, b, h0) -- the store-or-recompute
 * choice of the same section: a forward scan that keeps only the state
 * entering every 64-step chunk (in the workspace), then the backward kernel
 * rebuilds each chunk's states from it and b.
 *   a      [B, T, D] fp32   decays of the forward call
 *   b      [B, T, D] fp32   [opt] inputs of the forward call (required when h is NULL)
 *   h0     [B, D]    fp32   [opt] initial state of the forward call
 *   h      [B, T, D] fp32   [opt] states returned by the forward call (NULL = recompute)
 *   dh     [B, T, D] fp32   upstream gradient on every state
 *   dhT    [B, D]    fp32   [opt] upstream gradient on the returned h_T
 *   da, db [B, T, D] fp32   out
 *   dh0    [B, D]    fp32   [opt] out
 * Both h and b NULL is CLA_ERR_INVALID_ARG.  The workspace size query covers
 * the recompute path (it adds ceil(T/64) * B * D fp32 chunk states). */
int cla_scan_diag_bwd(const float *a, const float *b, const float *h0, const float *h,
                      const float *dh, const float *dhT, float *da, float *db,
                      float *dh0, int64_t B, int64_t T, int64_t D, void *ws,
                      size_t ws_bytes, void *stream);

/* Forward diagonal scan for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment variant of
 * cla_scan_diag_fwd.  It is meant for code that may not (or cannot) hand the
 * library a workspace: a plugin inside a framework that owns every device
 * allocation and offers no scratch buffer, a deployment whose device-memory
 * footprint is fixed ahead of time, or a path where an allocation call's
 * latency or implicit synchronisation is not allowed.  Inputs, outputs and
 * results are those of cla_scan_diag_fwd; the caller still passes every
 * input and output buffer.
 *  - Scratch: the look-back scratch lives in a 16 MiB array compiled into the
 *    library (one per GPU that loads it, held until the process exits).  No
 *    cudaMalloc, cudaFree or other allocating call is made.
 *  - Limit: sizes whose scratch exceeds 16 MiB are rejected with
 *    CLA_ERR_UNSUPPORTED and nothing is enqueued: about 89 million elements
 *    of B*T*D when D is a multiple of 4 (8 x 4096 x 1024 fits), about 22
 *    million otherwise.
 *  - Every call looks up the array's device address (cudaGetSymbolAddress)
 *    in the current device's context; the first lookup on a device may load
 *    the library's device code there, so make the first call on each device
 *    before any stream capture.
 *  - Every call shares the one array; the call clears what must start at
 *    zero.  Calls that overlap on the GPU (other streams, other host threads)
 *    race on it and must be serialised by the caller.
 *  - There is no workspace to pass to cla_check_status(): a look-back wait
 *    that gives up is reported by cla_scan_diag_noalloc_check_status(), until
 *    the next call clears it. */
int cla_scan_diag_fwd_noalloc(const float *a, const float *b, const float *h0,
                              float *h, float *hT, int64_t B, int64_t T,
                              int64_t D, void *stream);

/* Status of the last cla_scan_diag_fwd_noalloc call on the current device:
 * synchronises `stream` (the stream of that call), then reports
 * CLA_ERR_TIMEOUT if one of its look-back waits gave up, CLA_ERR_CUDA if the
 * stream holds an error, else CLA_OK.  Reads the static array's header into
 * host memory; allocates nothing.  The pages have no counterpart (a
 * deployment aid, as above). */
int cla_scan_diag_noalloc_check_status(void *stream);

/* ======================================================================== */
/* Selective (Mamba-1 style) diagonal scan                                  */
/* ======================================================================== */

/* Time steps between the states saved by the forward for the backward. */
#define CLA_SELECTIVE_CKPT_CHUNK 16

/* Bytes of workspace for cla_selective_scan_fwd / _bwd. */
size_t cla_selective_scan_workspace_size(int64_t B, int64_t T, int64_t D, int64_t N);

/* Elements of the checkpoint tensor [B, ceil(T/16), D, N] (fp32). */
size_t cla_selective_scan_ckpt_elems(int64_t B, int64_t T, int64_t D, int64_t N);

/* Forward: per channel d and state entry n, h_{t,d,n} = a h_{t-1,d,n} + b with
 * a = exp(delta_{t,d} A_{d,n}), b = delta_{t,d} Bm_t[n] x_{t,d}, and the read
 * y_{t,d} = sum_n Cm_t[n] h_{t,d,n} ("Parallel Scan", "When a scan is the
 * wrong tool": Mamba's selective decay; the (B, T, D, N) state never reaches
 * HBM).
 *   x      [B, T, D] bf16,  delta [B, T, D] fp32,  A [D, N] fp32
 *   Bm, Cm [B, T, N] bf16,  h0 [B, D, N] fp32 [opt]
 *   y      [B, T, D] fp32   out
 *   hT     [B, D, N] fp32   [opt] out
 *   ckpt   [B, ceil(T/16), D, N] fp32 [opt] out: the state entering every
 *          16-step interval, consumed by the backward
 * N must be 16 in this build. */
int cla_selective_scan_fwd(const uint16_t *x, const float *delta, const float *A,
                           const uint16_t *Bm, const uint16_t *Cm, const float *h0,
                           float *y, float *hT, float *ckpt, int64_t B, int64_t T,
                           int64_t D, int64_t N, void *ws, size_t ws_bytes,
                           void *stream);

/* Backward: the adjoint of every (d, n) recurrence with direct gradient
 * Cm_t[n] dy_{t,d}, recomputing the states from ckpt, then the chain rule
 * through a and b:
 *   dx_{t,d}     = sum_n hbar delta Bm_t[n]
 *   ddelta_{t,d} = sum_n hbar (h_{t-1} a A_{d,n} + Bm_t[n] x_{t,d})
 *   dA_{d,n}     = sum_{b,t} hbar h_{t-1} a delta
 *   dB_t[n]      = sum_d hbar delta x,    dC_t[n] = sum_d dy h_t
 *   dh0          = a_1 hbar_1
 *   ckpt   as written by the forward with the same inputs
 *   dy     [B, T, D] fp32;  dhT [B, D, N] fp32 [opt]
 *   dx     [B, T, D] fp32 out;  ddelta [B, T, D] fp32 out
 *   dA     [D, N] fp32 [opt] out;  dB, dC [B, T, N] fp32 out
 *   dh0    [B, D, N] fp32 [opt] out
 * Channel sums are reduced in a fixed order (no float atomics). */
int cla_selective_scan_bwd(const uint16_t *x, const float *delta, const float *A,
                           const uint16_t *Bm, const uint16_t *Cm, const float *h0,
                           const float *ckpt, const float *dy, const float *dhT,
                           float *dx, float *ddelta, float *dA, float *dB,
                           float *dC, float *dh0, int64_t B, int64_t T, int64_t D,
                           int64_t N, void *ws, size_t ws_bytes, void *stream);

/* ======================================================================== */
/* Chunkwise decayed linear attention (matrix state)                        */
/* ======================================================================== */

/* Bytes of workspace for cla_chunk_la_fwd / _bwd; 0 for sizes, head dims
 * or chunks those calls refuse. */
size_t cla_chunk_la_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                                   int64_t dim_v, int chunk);
/* The same query under the name the boundary's plan gives it. */
size_t cla_chunk_la_workspace(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                              int64_t dim_v, int chunk);

/* Forward of S_t = a_t S_{t-1} + k_t v_t^T (S is [dim_k, dim_v], rows indexed
 * by keys), o_t = S_t^T q_t, with a_t = exp(log_decay_t), computed chunkwise
 * ("Parallel Scan", "The chunkwise algorithm"; "Lightning Attention-2",
 * eqs. 8 and 10 and Algorithm 1, with per-token decays):
 *   O_[j] = (Q_[j] K_[j]^T . D) V_[j] + diag(lambda) Q_[j] S_[j-1]
 *   S_[j] = alpha_j S_[j-1] + K_[j]^T diag(gamma) V_[j]
 * D_rs = a_{t0+r:t0+s} (s <= r, unit diagonal), lambda_r = a_{t0+r:t0}
 * (includes the first token's decay), gamma_s = a_{t0+Tc:t0+s}
 * (gamma_Tc = 1); all from in-chunk sums of log_decay, never from long
 * cumulative sums or ratios ("Long products without underflow").  A decay of
 * exactly 0 (log_decay = -inf) is a reset and gives products of 0.  Decays
 * are gates in [0, 1], i.e. log_decay <= 0; larger values are computed as
 * given, but a product over up to 32 consecutive tokens beyond 2^127
 * overflows.
 *   q, k       [B, H, T, dim_k] bf16
 *   v          [B, H, T, dim_v] bf16
 *   log_decay  [B, H, T] fp32
 *   S0         [B, H, dim_k, dim_v] fp32 [opt]
 *   o          [B, H, T, dim_v] fp32 out (the accumulation precision: bf16
 *              rounding of the output alone would exceed the parity tolerance)
 *   ST         [B, H, dim_k, dim_v] fp32 [opt] out: S_T
 * Supported: dim_k and dim_v each in {64, 128}, chunk in {64, 128}; any
 * T >= 0 (the last chunk may be shorter). */
int cla_chunk_la_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const float *log_decay, const float *S0, float *o,
                     float *ST, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                     int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                     void *stream);

/* Backward ("Parallel Scan", "The backward pass of linear attention";
 * "Lightning Attention-2", eqs. 15, 17, 19, 20 and Algorithm 2, with the
 * decays above): a forward-order traversal rebuilds the chunk states and
 * gives dQ; a reverse-order traversal carries the adjoint state dS and gives
 * dK and dV; the decay gradient is the closed form
 *   dlog_decay_u = sum_{t>=u} q_t.dq_t - sum_{s>=u} k_s.dk_s + <dST, S_T>
 * (no per-token states), and dS0 is the adjoint state at t = 0.
 *   dO         [B, H, T, dim_v] bf16   upstream gradient on o
 *   dST        [B, H, dim_k, dim_v] fp32 [opt] upstream gradient on S_T
 *   dq, dk     [B, H, T, dim_k] fp32 out;  dv [B, H, T, dim_v] fp32 out
 *   dlog_decay [B, H, T] fp32 [opt] out;  dS0 [B, H, dim_k, dim_v] fp32 [opt] out
 * Same support as the forward. */
int cla_chunk_la_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const float *log_decay, const float *S0, const uint16_t *dO,
                     const float *dST, float *dq, float *dk, float *dv,
                     float *dlog_decay, float *dS0, int64_t B, int64_t H,
                     int64_t T, int64_t dim_k, int64_t dim_v, int chunk,
                     void *ws, size_t ws_bytes, void *stream);

/* Storing chunk states instead of rebuilding them ("Parallel Scan", "The
 * backward pass is a scan in reverse": the backward needs the forward's
 * states, which can be stored or recomputed from the inputs).  The library
 * splits each sequence into segments of chunks; the forward forms the state
 * entering every segment anyway, and the backward's forward-order traversal
 * (the one that gives dQ) needs exactly those states.
 *
 * Bytes of that checkpoint for these sizes: n_seg * B * H * dim_k * dim_v
 * fp32 values, n_seg fixed by the sizes and the chunk.  0 for sizes, head
 * dims or chunks the fwd / bwd calls refuse. */
size_t cla_chunk_la_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                              int64_t dim_v, int chunk);

/* cla_chunk_la_fwd that also writes the checkpoint: ckpt (device,
 * cla_chunk_la_ckpt_size bytes, 16-byte aligned, owned by the caller) gets
 * the state entering each segment.  ckpt = NULL is the plain forward.  When
 * T is shorter than one chunk nothing is written (the backward then rebuilds
 * its states itself). */
int cla_chunk_la_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const float *log_decay, const float *S0, float *o,
                          float *ST, float *ckpt, int64_t B, int64_t H, int64_t T,
                          int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                          size_t ws_bytes, void *stream);

/* cla_chunk_la_bwd that starts its forward-order traversal from the
 * checkpoint written by cla_chunk_la_fwd_ckpt with the same q, k, v,
 * log_decay, S0, sizes and chunk (read only; the results are those of
 * cla_chunk_la_bwd up to fp32 rounding).  ckpt = NULL rebuilds the states
 * (cla_chunk_la_bwd).  A checkpoint from other inputs gives wrong gradients;
 * nothing checks it. */
int cla_chunk_la_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const float *log_decay, const float *S0, const uint16_t *dO,
                          const float *dST, float *dq, float *dk, float *dv,
                          float *dlog_decay, float *dS0, const float *ckpt,
                          int64_t B, int64_t H, int64_t T, int64_t dim_k,
                          int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                          void *stream);

/* ======================================================================== */
/* Gated linear attention (matrix state, one decay per key dimension)       */
/* ======================================================================== */

/* Bytes of workspace for cla_gla_fwd; 0 for sizes, head dims or chunks that
 * call refuses. */
size_t cla_gla_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                              int64_t dim_v, int chunk);

/* Forward of S_t = diag(a_t) S_{t-1} + k_t v_t^T (S is [dim_k, dim_v], rows
 * indexed by keys; a_t = exp(log_decay_t) holds one decay per key
 * dimension), o_t = S_t^T q_t, computed chunkwise ("Parallel Scan", "What one
 * combine costs": a diagonal transition, and "The chunkwise algorithm": the
 * gated form S_t = G_t (.) S_{t-1} + k_t^T v_t).  With c the in-chunk
 * cumulative log2 decays and m a chunk's 32nd token, the decay between a
 * read at r and a write at s factors as 2^(c_r - c_m) 2^(c_m - c_s), so the
 * queries and keys are scaled per element and the intra-chunk scores are one
 * product, masked causally:
 *   O_[j]  = ((Q~ K~^T) . M) V_[j] + Q~ diag(2^c_m) S_[j-1]
 *   S_[j]  = diag(2^(c_L - c_m)) (diag(2^c_m) S_[j-1] + K~^T V_[j])
 * with Q~ = Q (.) 2^(c - c_m), K~ = K (.) 2^(c_m - c).
 *   q, k       [B, H, T, dim_k] bf16
 *   v          [B, H, T, dim_v] bf16
 *   log_decay  [B, H, T, dim_k] fp32 (natural log of the gates, <= 0)
 *   S0         [B, H, dim_k, dim_v] fp32 [opt]
 *   o          [B, H, T, dim_v] fp32 out
 *   ST         [B, H, dim_k, dim_v] fp32 [opt] out: S_T
 * Supported: dim_k 64 or 128, dim_v a multiple of 64 up to 1024, chunk 64,
 * any T >= 0.  Range: in every key dimension of every 64-token chunk, the
 * gate product over the chunk's first 32 tokens and over its last 32 must be
 * at least 2^-120 (no zero gates); the kernel checks this on the device and a
 * violation makes cla_check_status(ws, stream) return CLA_ERR_UNSUPPORTED
 * (the call's outputs are then not valid). */
int cla_gla_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                const float *log_decay, const float *S0, float *o, float *ST,
                int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                int chunk, void *ws, size_t ws_bytes, void *stream);

/* Bytes of workspace for cla_gla_bwd (look-back arrays, the decay
 * gradient's partial sums and, when the dV and dK traversals get the same
 * segments of chunks, the adjoint state entering each segment, which the dV
 * traversal saves and the dK traversal starts from); 0 for sizes, head dims
 * or chunks that call refuses. */
size_t cla_gla_bwd_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                                  int64_t dim_v, int chunk);

/* Backward of cla_gla_fwd ("Parallel Scan", "The backward pass of linear
 * attention", with the scalar decay replaced by the diagonal one, and the
 * closed-form decay gradient per key dimension of Yang et al. that the
 * section cites):
 *   dQ  a forward-order traversal that rebuilds the states from S0;
 *   dV, dS0  the forward kernel run on the reversed adjoint recursion
 *       Sbar_t = q_t^T dO_t + diag(a_{t+1}) Sbar_{t+1} (from dST);
 *   dK  a reverse-order traversal carrying the adjoint state;
 *   dlog_decay_u[i] = sum_{t>=u} (q_t[i] dq_t[i] - k_t[i] dk_t[i])
 *                     + sum_j dST[i][j] S_T[i][j]
 * (no per-token states).  The decay of the query and key gradients sits on
 * their own column, dq_r[i] = 2^(c_r - c_m)[i] (((dO V^T) . M) K~ + dO S'^T)
 * [r][i], with the same midpoint factoring as the forward.
 *   dO          [B, H, T, dim_v] bf16   upstream gradient on o
 *   dST         [B, H, dim_k, dim_v] fp32 [opt] upstream gradient on S_T
 *   dq, dk      [B, H, T, dim_k] fp32 out;  dv [B, H, T, dim_v] fp32 out
 *   dlog_decay  [B, H, T, dim_k] fp32 [opt] out;  dS0 [B, H, dim_k, dim_v] fp32 [opt] out
 * Supported: dim_k and dim_v 64 or 128, chunk 64; the forward's decay range
 * (reported the same way through cla_check_status). */
int cla_gla_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                const float *log_decay, const float *S0, const uint16_t *dO,
                const float *dST, float *dq, float *dk, float *dv,
                float *dlog_decay, float *dS0, int64_t B, int64_t H, int64_t T,
                int64_t dim_k, int64_t dim_v, int chunk, void *ws, size_t ws_bytes,
                void *stream);

/* The GLA checkpoint ("Parallel Scan", "The backward pass is a scan in
 * reverse": store the states or recompute them).  Every traversal of a head's
 * sequence splits it into the same segments of chunks; the forward forms the
 * state entering every segment, and the backward's forward-order traversal
 * (the one that gives dq) needs exactly those states.  Bytes of the
 * checkpoint: n_seg * B * H * dim_k * dim_v fp32 values, n_seg fixed by the
 * sizes; 0 for sizes, head dims or chunks the fwd / bwd calls refuse. */
size_t cla_gla_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                         int64_t dim_v, int chunk);

/* cla_gla_fwd that also writes the checkpoint: ckpt (device,
 * cla_gla_ckpt_size bytes, 16-byte aligned, owned by the caller) gets the
 * state entering each segment, [n_seg][B * H][dim_k][dim_v].  ckpt = NULL is
 * the plain forward; a checkpoint needs dim_k and dim_v of 64 or 128 (what
 * the backward takes). */
int cla_gla_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const float *log_decay, const float *S0, float *o, float *ST,
                     float *ckpt, int64_t B, int64_t H, int64_t T, int64_t dim_k,
                     int64_t dim_v, int chunk, void *ws, size_t ws_bytes, void *stream);

/* cla_gla_bwd whose dq traversal starts every segment from the checkpoint a
 * cla_gla_fwd_ckpt call on the same q, k, v, log_decay, S0, sizes and chunk
 * wrote (read only), instead of re-forming those states; the results are
 * those of cla_gla_bwd up to fp32 rounding.  ckpt = NULL is cla_gla_bwd.  A
 * checkpoint from other inputs gives wrong gradients; nothing checks it. */
int cla_gla_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const float *log_decay, const float *S0, const uint16_t *dO,
                     const float *dST, float *dq, float *dk, float *dv,
                     float *dlog_decay, float *dS0, const float *ckpt, int64_t B,
                     int64_t H, int64_t T, int64_t dim_k, int64_t dim_v, int chunk,
                     void *ws, size_t ws_bytes, void *stream);

/* ======================================================================== */
/* Delta rule with a decay per head (Gated DeltaNet)                         */
/* ======================================================================== */

/* Bytes of workspace for cla_delta_fwd: its 256-byte header (the error flag)
 * and room for every chunk's (I + A)^-1 (B H ceil(T / 64) x 16 KB: two bf16
 * parts of the 64 x 64 matrix), which the call then forms for all chunks at
 * once before the chunk loop; 0 for sizes, head dims or chunks that call
 * refuses.  cla_delta_fwd also accepts a header-only workspace (256 bytes):
 * the chunk loop then forms each (I + A)^-1 itself, with the same result
 * bits, more slowly. */
size_t cla_delta_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                                int64_t dim_v, int chunk);

/* Forward of S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
 * o_t = S_t^T q_t ("Parallel Scan", "What one combine costs": a transition
 * that is the identity minus a rank-one matrix, overwriting what the state
 * stores under a key, and its WY representation; "At real scale": the Gated
 * DeltaNet layer's decay per head), chunkwise: inside a 64-token chunk with
 * cumulative decays gamma and A_rs = beta_r (gamma_r / gamma_s) k_r . k_s
 * (s < r),
 *   Veff = (I + A)^-1 diag(beta) (V - diag(gamma) K S)
 *   O    = diag(gamma) Q S + ((Q K^T) . D) Veff
 *   S'   = gamma_L S + K^T diag(gamma_L / gamma) Veff.
 * The chunks of a head run in order (one block per head and 64 value
 * columns).
 *   q, k       [B, H, T, dim_k] bf16 (keys are used as given; the layer
 *              normally L2-normalises them)
 *   v          [B, H, T, dim_v] bf16
 *   log_decay  [B, H, T] fp32 (natural log of a_t, finite)
 *   beta       [B, H, T] fp32 (write strengths, finite)
 *   S0         [B, H, dim_k, dim_v] fp32 [opt]
 *   o          [B, H, T, dim_v] fp32 out;  ST [B, H, dim_k, dim_v] fp32 [opt] out
 * Supported: dim_k 64 or 128, dim_v a multiple of 64 up to 1024, chunk 64.
 * A non-finite log decay or beta makes cla_check_status(ws, stream) return
 * CLA_ERR_UNSUPPORTED (the outputs are then not valid). */
int cla_delta_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *log_decay, const float *beta, const float *S0,
                  float *o, float *ST, int64_t B, int64_t H, int64_t T,
                  int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                  size_t ws_bytes, void *stream);

/* Bytes of workspace for cla_delta_bwd: the header, the state entering every
 * chunk (B H ceil(T / 64) dim_k dim_v fp32), every chunk's (I + A)^-1 as two
 * bf16 parts and its E = A without the gate strengths (fp32), together
 * B H ceil(T / 64) x 32 KB, and, for dim_v > 64, partial
 * key-side gradients of the value-column blocks after the first
 * ((dim_v / 64 - 1) B H T (2 dim_k + 2) fp32); 0 for sizes, head dims or
 * chunks that call refuses.  cla_delta_bwd_ckpt needs this less
 * cla_delta_ckpt_size (the checkpoint holds the states, the inverses and E). */
size_t cla_delta_bwd_workspace_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                                    int64_t dim_v, int chunk);

/* Backward of cla_delta_fwd: the adjoint of the chunk form ("Parallel Scan",
 * "What one combine costs" for the transition and its WY factors; "The
 * backward pass is a scan in reverse" for the adjoint carried from the last
 * chunk to the first).  A states pass of the forward kernel writes the state
 * S entering every chunk; then, chunks in reverse with dS' the adjoint of the
 * state leaving the chunk, U = Veff, w_r = gamma_L / gamma_r:
 *   dU = P^T dO + diag(w) K dS',  dX = (I + A)^-T dU,  dV = diag(beta) dX
 *   dP = dO U^T (s <= r),  dA = -dX U^T (s < r),  F = diag(beta) dA . D
 *   dQ = (dP . D) K + diag(gamma) dO S^T
 *   dK = (dP . D)^T Q + (F + F^T) K + diag(w) U dS'^T - diag(beta gamma) dX S^T
 *   dbeta_r = (V - diag(gamma) K S)_r . dX_r + sum_s dA_rs D_rs k_r . k_s
 *   dS = gamma_L dS' + Q^T diag(gamma) dO - K^T diag(beta gamma) dX
 * and dlog_decay the in-chunk suffix sums of the gradient on the cumulative
 * log decays.
 *   dO          [B, H, T, dim_v] bf16   upstream gradient on o
 *   dST         [B, H, dim_k, dim_v] fp32 [opt] upstream gradient on S_T
 *   dq, dk      [B, H, T, dim_k] fp32 out;  dv [B, H, T, dim_v] fp32 out
 *   dlog_decay, dbeta [B, H, T] fp32 out;  dS0 [B, H, dim_k, dim_v] fp32 [opt] out
 * Supported and checked as cla_delta_fwd; dq, dk, dv, dS0, dST and S0 8-byte
 * aligned.  A non-finite log decay or beta is reported through
 * cla_check_status(ws, stream) as in the forward. */
int cla_delta_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *log_decay, const float *beta, const float *S0,
                  const uint16_t *dO, const float *dST, float *dq, float *dk,
                  float *dv, float *dlog_decay, float *dbeta, float *dS0,
                  int64_t B, int64_t H, int64_t T, int64_t dim_k, int64_t dim_v,
                  int chunk, void *ws, size_t ws_bytes, void *stream);

/* Checkpoint of the delta rule's forward for its backward ("The backward pass
 * is a scan in reverse": store the states or recompute them).  The backward
 * works from the state entering every chunk; the forward computes exactly
 * those states, so it can save them instead of the backward re-running it.
 * The checkpoint also keeps every chunk's (I + A)^-1 and E (A without the
 * gate strengths; both depend on k, log_decay and beta only), so the backward
 * reads them instead of re-forming them.  Bytes of the checkpoint:
 * B H ceil(T / 64) dim_k dim_v fp32 values (rounded up to 16 bytes), then
 * B H ceil(T / 64) x 16 KB of inverse parts and B H ceil(T / 64) x 16 KB of E;
 * 0 for sizes, head dims or chunks the fwd / bwd calls refuse. */
size_t cla_delta_ckpt_size(int64_t B, int64_t H, int64_t T, int64_t dim_k,
                           int64_t dim_v, int chunk);

/* cla_delta_fwd that also writes the checkpoint: ckpt (device,
 * cla_delta_ckpt_size bytes, 16-byte aligned, owned by the caller) gets the
 * state entering each 64-token chunk, [B, H, ceil(T / 64), dim_k, dim_v],
 * followed by each chunk's (I + A)^-1 parts and E (the forward then needs
 * only the workspace's header).
 * ckpt = NULL is the plain forward. */
int cla_delta_fwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *log_decay, const float *beta, const float *S0,
                       float *o, float *ST, float *ckpt, int64_t B, int64_t H,
                       int64_t T, int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                       size_t ws_bytes, void *stream);

/* cla_delta_bwd from the checkpoint a cla_delta_fwd_ckpt call on the same q,
 * k, v, log_decay, beta, S0, sizes and chunk wrote (read only): no states
 * pass, and the workspace needs only the header and the partial gradients
 * (cla_delta_bwd_workspace_size bytes are always enough).  The gradients are
 * those of cla_delta_bwd (the same states, bit for bit).  ckpt = NULL is
 * cla_delta_bwd.  A checkpoint from other inputs gives wrong gradients;
 * nothing checks it, and the non-finite input check ran in the forward. */
int cla_delta_bwd_ckpt(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *log_decay, const float *beta, const float *S0,
                       const uint16_t *dO, const float *dST, float *dq, float *dk,
                       float *dv, float *dlog_decay, float *dbeta, float *dS0,
                       const float *ckpt, int64_t B, int64_t H, int64_t T,
                       int64_t dim_k, int64_t dim_v, int chunk, void *ws,
                       size_t ws_bytes, void *stream);

/* ======================================================================== */
/* State passing between slices of one sequence                             */
/* ======================================================================== */

/* Total decay of a slice ("Parallel Scan", "Splitting one sequence across
 * devices": each device's pair holds its slice's product of decays):
 *   alpha[bh][a] = exp(sum_t log_decay[bh][t][a])
 *   log_decay  [BH, T, A] fp32 (A = 1: one decay per head, as chunk_la's
 *              [B, H, T]; A = dim_k: gated decays, as gla's [B, H, T, dim_k])
 *   alpha      [BH, A] fp32 out (0 where the slice holds a reset). */
int cla_decay_total(const float *log_decay, float *alpha, int64_t BH, int64_t T,
                    int64_t A, void *stream);

/* The state entering a slice, from the pairs (alpha_j, dS_j) of the slices
 * before it (same section; the combine (a1, b1) . (a2, b2) = (a1 a2,
 * a2 b1 + b2) of "The scan for one number of state"):
 *   out = fold over c = 0..count-1, j = first + c * step, of
 *         acc <- diag(alpha_j) acc + dS_j,  from acc = edge (0 if NULL).
 *   alpha  [P, BH, A] fp32: A = 1 scales a head's whole state, A > 1 scales
 *          state row r by alpha[.][.][r / (n / A)] (one decay per key row)
 *   dS     [P, BH, n] fp32 (n = dim_k * dim_v state entries, rows first)
 *   edge   [BH, n] fp32 [opt]: the initial state (forward) or the upstream
 *          gradient of the final state (backward, composed from the right
 *          with step = -1)
 *   out    [BH, n] fp32 out
 * n must be a multiple of A; pair indices must lie in [0, P). */
int cla_state_compose(const float *alpha, const float *dS, const float *edge,
                      float *out, int64_t P, int64_t BH, int64_t n, int64_t A,
                      int64_t first, int64_t count, int64_t step, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CLA_H_ */
