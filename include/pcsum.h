/*
 * pcsum.h - C ABI of the GB300 log-space sum-layer library (libpcsum.so).
 *
 * What it computes
 * ----------------
 * The dense sum layer of a probabilistic circuit, in log space, and the circuits
 * built from it (pyjuice pull request #62, "precision option / dense sum layers
 * through cuBLAS / fp32 backward on tensor cores", Summary 2 and 3):
 *
 *   forward    out[i,b] = m_b + log sum_j theta[i,j] * exp(x[j,b] - m_b)
 *              m_b = max_j x[j,b], the per-sample maximum over the group's children
 *   element    e[j,b]   = sum_i theta[i,j] * f[i,b] * exp(x[j,b] - out[i,b])
 *   parameter  F[i,j]   = theta[i,j] * sum_b f[i,b] * exp(x[j,b] - out[i,b])
 *
 * and the LowRank "exp_sum" per-sample scale (pyjuice.parameterizations.LowRank
 * API doc, intro formulas and Training):
 *   theta_b[i,j] = theta[i,j] * exp((A_b B_b)[i,j]) / Z_b[i].
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every array argument is DEVICE memory owned by the caller, unless its comment
 *   says HOST. The library never allocates device memory: scratch comes from the
 *   caller's workspace `ws` of at least the size the matching *_workspace query
 *   reports (16-byte aligned). float arrays are float32, row-major (C order).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream), perform no host synchronisation and allocate nothing.
 * - Arguments are validated before anything is launched. On failure the call
 *   returns a status other than PC_OK, launches nothing and leaves a one-line
 *   reason in pc_last_error() (thread-local). PC_ERR_CUDA reports a CUDA launch
 *   error; device-side waits are bounded and a timed-out kernel records
 *   PC_ERR_TIMEOUT in a device status word read by pc_device_status().
 * - Precision (pyjuice PR #62, Summary 1 table) selects how the products of the
 *   contractions are formed; accumulation is always float32 in tensor memory:
 *     PC_PREC_AUTO  bfloat16 operands (round to nearest even)
 *     PC_PREC_TF32  TF32 operands (round to nearest, ties away from zero)
 *     PC_PREC_FP32  three TF32 products hi*hi + hi*lo + lo*hi (fp32-level)
 *   Any other value returns PC_ERR_UNKNOWN_PRECISION, naming the valid modes.
 * - Flow outputs are overwritten, or added to when `accumulate` != 0.
 */
#ifndef PCSUM_H_
#define PCSUM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PCSUM_API __attribute__((visibility("default")))
#else
#define PCSUM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pc_stream_t;

typedef enum {
  PC_PREC_AUTO = 0, /* bf16 products */
  PC_PREC_TF32 = 1, /* TF32 products */
  PC_PREC_FP32 = 2  /* 3xTF32 products */
} pc_precision_t;

typedef enum {
  PC_OK = 0,
  PC_ERR_NULL = 1,              /* a required pointer is NULL */
  PC_ERR_SHAPE = 2,             /* a size is out of range or inconsistent */
  PC_ERR_ALIGNMENT = 3,         /* a pointer is not 16-byte aligned */
  PC_ERR_UNKNOWN_PRECISION = 4, /* precision is not one of pc_precision_t */
  PC_ERR_WORKSPACE = 5,         /* workspace NULL or smaller than the query's size */
  PC_ERR_UNSUPPORTED = 6,       /* a valid request outside the library's limits */
  PC_ERR_CUDA = 7,              /* a CUDA call failed (launch or device query) */
  PC_ERR_TIMEOUT = 8,           /* a device-side wait ran out (see pc_device_status) */
  PC_ERR_RANGE = 9              /* an HMM sample left the exactly-scaled range (see pc_hmm_fwd_bwd) */
} pc_status_t;

/* Library version string, e.g. "pcsum 0.1 sm_103a". Static storage. */
PCSUM_API const char* pc_version(void);

/* Static English name of a status code. */
PCSUM_API const char* pc_status_string(pc_status_t status);

/* Detail of the last failing call on this host thread ("" if none). Valid until the
 * next call into the library from the same thread. */
PCSUM_API const char* pc_last_error(void);

/* Number of kernels this library has launched in the process so far (all entry
 * points, all devices). */
PCSUM_API unsigned long long pc_launch_count(void);

/* Synchronises `stream`, then reads and clears the device status word of the current
 * device. Returns PC_OK; PC_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * read; else PC_ERR_RANGE if an HMM call flagged a sample whose values left the range its
 * per-layer scaling keeps exact (that sample's LL is NaN and it passed no flow); or
 * PC_ERR_CUDA. Diagnostic; not for the hot path. */
PCSUM_API pc_status_t pc_device_status(pc_stream_t stream);

/* Limit, in nanoseconds, of the first waits of the tensor-core contraction kernel on the
 * current device (a free ring slot, a filled slot, a free or complete accumulator);
 * 0 restores the default of 2 s. A kernel whose wait runs out records PC_ERR_TIMEOUT
 * for pc_device_status, skips the rest of its tile and exits cleanly: waits for work it
 * has already issued (copies landing, MMAs completing before tensor memory is freed)
 * always keep the default limit, so no copy or MMA is left in flight. The limit is a
 * device-wide watchdog setting for failure detection and its tests: a limit shorter
 * than a tile's K loop makes calls give up and return garbage outputs. Synchronous
 * (a host-to-device copy); takes effect for kernels launched after it returns; call it
 * while no library kernel is running. Errors: PC_ERR_CUDA. */
PCSUM_API pc_status_t pc_set_wait_limit_ns(unsigned long long ns);

/* Timing of the tensor-core contractions, for measurement. Between
 * pc_profile_start(capacity) and pc_profile_stop, every contraction the library
 * launches records a CUDA event pair on its stream (at most `capacity` records), except
 * the HMM's chain contractions: each chain of T-1 consecutive launches of one kind is
 * one record (events between them would break their programmatic overlap).
 * pc_profile_stop synchronises the device, then writes for each record i
 * (i < *count <= capacity): ms[i] = elapsed device time, kind[i] = which contraction
 * (PC_KIND_*), flops[i] = the algorithmic flops of its launches, 2*M*N*K each (each
 * product counted once), launches[i] = how many launches the record spans. For the
 * memory-bound kinds (PC_KIND_EM_MSTEP and the *_MEM kinds: every launch of the HMM and
 * HCLT calls that is not a contraction, i.e. operand copies and transposes, emission
 * gathers, product layers, root and scaled flows, token buckets and dE gathers) flops[i]
 * holds the launch's algorithmic bytes instead (each input read once, each output written
 * once). Any output pointer may be NULL. Not thread-safe; host-side event objects only,
 * no device memory. */
typedef enum {
  PC_KIND_LAYER_FWD = 0, PC_KIND_LAYER_ELEM = 1, PC_KIND_LAYER_PARAM = 2,
  PC_KIND_HMM_FWD = 3, PC_KIND_HMM_ELEM = 4, PC_KIND_HMM_PARAM = 5,
  PC_KIND_HCLT_FWD = 6, PC_KIND_HCLT_ELEM = 7, PC_KIND_HCLT_PARAM = 8,
  PC_KIND_LOWRANK_FWD = 9, PC_KIND_LOWRANK_BWD = 10, PC_KIND_EM_MSTEP = 11,
  PC_KIND_HMM_MEM = 12, PC_KIND_HCLT_MEM = 13
} pc_kind_t;
PCSUM_API pc_status_t pc_profile_start(int capacity);
PCSUM_API pc_status_t pc_profile_stop(int* count, float* ms, int* kind, long long* flops,
                                      int* launches, int capacity);

/* ------------------------------------------------------------------------------
 * Dense sum layer, G groups (pyjuice PR #62, Summary 2: shared-children layers
 * and evenly strided child groups run as batched GEMMs; Summary 3: the element-
 * and parameter-flow contractions).
 *
 *   theta [G][M][N]   parameters of group g (row i = node, column j = child).
 *   x     [R][B]      child log-values, one row of B samples per child; group g's
 *                     children are rows g*child_stride .. g*child_stride+N-1.
 *                     G == 1: any child_stride (0 is the shared-children layout).
 *                     G > 1: child_stride >= N (non-overlapping groups).
 *   out   [G][M][B]   node log-values. -inf where the sum is 0 or every child is -inf.
 *   f     [G][M][B]   node flows (backward input).
 *   e     like x      element flows; rows outside every group are not touched.
 *                     NULL = not computed.
 *   F     [G][M][N]   parameter flows. NULL = not computed.
 * Limits: 1 <= G <= 65535; 1 <= M, N, B < 2^24; x and the arrays above hold at
 * most 2^31 rows. Scratch: pc_sum_layer_workspace (covers both directions).
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_sum_layer_workspace(int G, int M, int N, int B, pc_precision_t prec,
                                   size_t* bytes);

PCSUM_API pc_status_t pc_sum_layer_fwd(int G, int M, int N, int B, const float* theta, const float* x,
                             long long child_stride, float* out, pc_precision_t prec,
                             void* ws, size_t ws_bytes, pc_stream_t stream);

PCSUM_API pc_status_t pc_sum_layer_bwd(int G, int M, int N, int B, const float* theta, const float* x,
                             long long child_stride, const float* out, const float* f,
                             float* e, float* F, int accumulate, pc_precision_t prec,
                             void* ws, size_t ws_bytes, pc_stream_t stream);

/* pc_sum_layer_fwd for callers that cannot allocate device memory. The pages have no
 * counterpart to this entry point; it exists because some callers can neither call
 * cudaMalloc nor hand over a workspace: a plugin whose host framework owns all device
 * memory and exposes no allocator, or a hot path where an allocation (and the
 * synchronisation it brings) is not allowed. Same arguments and results as
 * pc_sum_layer_fwd, without ws / ws_bytes: the scratch is a 16 MiB array built into
 * the library, held on every GPU that loads it until the process exits.
 *   - Requests whose scratch (pc_sum_layer_workspace) exceeds 16 MiB return
 *     PC_ERR_UNSUPPORTED with the sizes in pc_last_error(); nothing is launched.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call uses the same array: calls that may overlap on the GPU (different
 *     streams, concurrent graph launches) race and must be serialised by the caller.
 *     Nothing in the array needs to start at zero; each call writes what it reads. */
PCSUM_API pc_status_t pc_sum_layer_fwd_noalloc(int G, int M, int N, int B, const float* theta,
                                               const float* x, long long child_stride, float* out,
                                               pc_precision_t prec, pc_stream_t stream);

/* ------------------------------------------------------------------------------
 * Whole HMM circuit, forward + backward (pyjuice PR #62, Results table "HMM, 4096
 * latents, 32 positions"; Summary 2, first bullet: its layers share their children).
 * The circuit is P(x) = sum_z pi(z_1) prod_t E(z_t, x_t) prod_t A(z_t, z_{t+1}),
 * built from the last position back as T-1 tied H x H sum layers with product
 * (emission) layers between them and a root sum layer over pi.
 *
 *   tokens [B][T] int32 in [0, V)           observed sequence of each sample
 *   pi [H], A [H][H] (A[k][l] = P(z_{t+1}=l | z_t=k)), E [H][V]  (non-negative)
 *   ll [B] double                           log P(x) per sample (written)
 *   dpi [H], dA [H][H], dE [H][V]           EM flows summed over the batch (posterior
 *                                           expected counts); each may be NULL. When
 *                                           all three are NULL only ll is computed.
 * Limits: 1 <= H <= 16384, 1 <= T <= 4096, 1 <= V <= 65536, 1 <= B <= 65536.
 * Tokens outside [0, V) are undefined behaviour. Numerical range: every layer scales
 * a sample's values by 1 / (max_k E[k,x_t] * sum_l A[k,l] times the previous position's
 * maximum) (at most 2^100), an upper bound of the largest value, and the per-sample
 * log-offsets accumulate in double; exact zeros (in E, A or pi) give exact zeros, and a
 * sequence of probability 0 gets ll = -inf and passes no flow. The results are exact
 * (to the mode's rounding) while at every position the largest scaled value stays
 * above 2^-80, i.e. the bound is looser than e^-55 nowhere. A sample for which that
 * fails is flagged instead of returning a wrong value: its ll is NaN, it passes no
 * flow (the other samples' flows are unaffected) and pc_device_status reports
 * PC_ERR_RANGE.
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_hmm_workspace(int H, int T, int V, int B, pc_precision_t prec, size_t* bytes);

PCSUM_API pc_status_t pc_hmm_fwd_bwd(int H, int T, int V, int B, const int32_t* tokens, const float* pi,
                           const float* A, const float* E, double* ll, float* dpi, float* dA,
                           float* dE, int accumulate, pc_precision_t prec, void* ws,
                           size_t ws_bytes, pc_stream_t stream);

/* ------------------------------------------------------------------------------
 * Whole HCLT circuit, forward + backward (pyjuice PR #62, Results table "HCLT, 1024
 * latents, 768 variables, 512 categories"; Summary 2, second bullet: its layers run
 * as batched GEMMs over evenly strided child groups). A latent tree over the
 * variables:  n_v(z) = E_v[z, x_v] prod_{c: parent[c]=v} sum_{z'} W_c[z,z'] n_c(z'),
 * LL = log sum_z pi[z] n_0(z). Edges are processed level by level (one grouped
 * contraction per level of equal child height).
 *
 *   parent [nvars] int32 HOST     parent[0] = -1, parent[i] in [0, i)
 *   data   [B][nvars] int32       category of each variable per sample, in [0, C)
 *                                 (a category outside [0, C) has emission 0)
 *   pi [H], W [nvars][H][H] (W[c][z_parent][z_c]; W[0] unused), E [nvars][H][C]
 *   ll [B] double                 log P(x) per sample (written)
 *   dpi [H], dW [nvars][H][H] (dW[0] = 0), dE [nvars][H][C]   EM flows summed over
 *                                 the batch; each may be NULL; all NULL = ll only.
 * Limits: 1 <= nvars <= 65535, 1 <= H <= 8192, 1 <= C <= 8192, 1 <= B <= 65535.
 * The tree plan the call derives from `parent` (a few KB) reaches the device inside
 * kernel arguments, not through a host-to-device copy, so the call can be captured
 * into a CUDA graph like the others; a captured graph replays the tree it was
 * captured with.
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_hclt_workspace(int nvars, int H, int C, int B, pc_precision_t prec,
                                        size_t* bytes);

PCSUM_API pc_status_t pc_hclt_fwd_bwd(int nvars, int H, int C, int B, const int32_t* parent,
                                      const int32_t* data, const float* pi, const float* W,
                                      const float* E, double* ll, float* dpi, float* dW, float* dE,
                                      int accumulate, pc_precision_t prec, void* ws,
                                      size_t ws_bytes, pc_stream_t stream);

/* The HCLT's parameters prepared once for many calls. Within an EM iteration every batch
 * reads the same W and E, and pc_hclt_fwd_bwd converts them on every call into the
 * formats its contractions read: W's per-edge operand copy in the tree's level order and
 * its transpose (2 x nvars x H x H values) and E transposed per variable. With
 * pc_hclt_prepare run once after the parameters change, pc_hclt_fwd_bwd_prepared skips
 * those conversions and computes the same results as pc_hclt_fwd_bwd.
 *
 * pc_hclt_prepare_bytes: the size of the prepared buffer for the tree size, H, C and
 *   precision (errors as pc_hclt_workspace).
 * pc_hclt_prepare: writes the prepared buffer `prep` (caller-owned device memory of at
 *   least that size) from parent (HOST, as for pc_hclt_fwd_bwd), W and E; asynchronous
 *   on `stream`, capturable. Errors: PC_ERR_NULL, PC_ERR_SHAPE (sizes or parent),
 *   PC_ERR_WORKSPACE (prep NULL or too small), PC_ERR_UNKNOWN_PRECISION.
 * pc_hclt_prepared_workspace: the workspace of pc_hclt_fwd_bwd_prepared (smaller than
 *   pc_hclt_workspace's by the prepared data).
 * pc_hclt_fwd_bwd_prepared: pc_hclt_fwd_bwd with `prep` in place of E. W is still read
 *   (the parameter flows are W times the contraction). `prep` must have been written by
 *   pc_hclt_prepare for the same parent, W, E, sizes and precision, and W and E must not
 *   have changed since: the library cannot check that without reading device memory. */
PCSUM_API pc_status_t pc_hclt_prepare_bytes(int nvars, int H, int C, pc_precision_t prec, size_t* bytes);
PCSUM_API pc_status_t pc_hclt_prepare(int nvars, int H, int C, const int32_t* parent, const float* W,
                                      const float* E, pc_precision_t prec, void* prep, size_t prep_bytes,
                                      pc_stream_t stream);
PCSUM_API pc_status_t pc_hclt_prepared_workspace(int nvars, int H, int C, int B, pc_precision_t prec,
                                                 size_t* bytes);
PCSUM_API pc_status_t pc_hclt_fwd_bwd_prepared(int nvars, int H, int C, int B, const int32_t* parent,
                                               const int32_t* data, const float* pi, const float* W,
                                               const void* prep, size_t prep_bytes, double* ll, float* dpi,
                                               float* dW, float* dE, int accumulate, pc_precision_t prec,
                                               void* ws, size_t ws_bytes, pc_stream_t stream);

/* ------------------------------------------------------------------------------
 * LowRank "exp_sum" per-sample scale on a dense sum layer with shared children
 * (pyjuice LowRank API doc: intro formulas, Tensor layout, Training, Note). Per sample b
 *   S_b = A_b B_b,  g_b = exp(S_b),  Z_b[i] = sum_j theta[i,j] g_b[i,j],
 *   theta_b = theta g_b / Z_b,       out[i,b] = log sum_j theta_b[i,j] exp(x[j,b]).
 * The per-sample scale is made on the tensor cores tile by tile and never stored.
 *
 *   theta [M][N]                shared parameters (rows need not sum to 1)
 *   A [B][M][K], Bm [B][K][N]   the factors, K = rank, 1 <= K <= 64
 *   x [N][B]                    child log-values
 *   out [M][B]                  node log-values (written)
 *   logZ [B][M]                 log Z_b[i] (written by the forward, read by the backward)
 * Backward for node flows f [M][B], with p = theta_b exp(x_j - out_i), q = theta_b:
 *   dA [B][M][K] = D B_b^T and dB [B][K][N] = A_b^T D with D = f (p - q), the gradient
 *   of sum f out; e [N][B] = sum_i f p (element flows); Fplus [M][N] = sum_b f p
 *   (parameter flows F+); Wstat [M][N] = sum_b f g_b / Z_b (the Z-correction statistic,
 *   F- = theta Wstat). Each output may be NULL (Wstat NULL = no Z correction); with
 *   accumulate != 0 the results are added to the outputs. Every output element is
 *   written by one thread: the results are deterministic.
 * Precision: S from bf16 hi + lo products (auto), one TF32 pass (tf32) or 3xTF32 (fp32);
 * the gradient contractions one bf16 term (auto), TF32, or 3xTF32.
 * Limits: K <= 64 (PC_ERR_UNSUPPORTED above), B <= 65535. M, N or B may be 0.
 * Workspace: pc_lowrank_exp_sum_workspace(..., with_backward, ...) bytes, 16-byte aligned.
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_lowrank_exp_sum_workspace(int M, int N, int K, int B, int with_backward,
                                                   pc_precision_t prec, size_t* bytes);

PCSUM_API pc_status_t pc_lowrank_exp_sum_fwd(int M, int N, int K, int B, const float* theta,
                                             const float* A, const float* Bm, const float* x,
                                             float* out, float* logZ, pc_precision_t prec,
                                             void* ws, size_t ws_bytes, pc_stream_t stream);

PCSUM_API pc_status_t pc_lowrank_exp_sum_bwd(int M, int N, int K, int B, const float* theta,
                                             const float* A, const float* Bm, const float* x,
                                             const float* out, const float* logZ, const float* f,
                                             float* dA, float* dB, float* e, float* Fplus,
                                             float* Wstat, int accumulate, pc_precision_t prec,
                                             void* ws, size_t ws_bytes, pc_stream_t stream);

/* ------------------------------------------------------------------------------
 * LowRank "sum_exp" per-sample scale (pyjuice LowRank API doc: intro formulas, the second
 * form of the scale; Note: "sum_exp" through the plain sum-layer kernels on a virtual
 * batch). Per sample b
 *   g_b[i,j] = sum_r exp(A_b[i,r]) exp(B_b[r,j]),  Z_b[i] = sum_j theta[i,j] g_b[i,j],
 *   theta_b = theta g_b / Z_b,                     out[i,b] = log sum_j theta_b[i,j] exp(x[j,b]).
 * Arguments, layouts and outputs as for "exp_sum" above (theta [M][N], A [B][M][K],
 * Bm [B][K][N], x [N][B], out [M][B], logZ [B][M]; backward for node flows f [M][B]: dA,
 * dB = the gradients of sum f out, e, Fplus, Wstat, each optional, accumulate adds). The
 * backward recomputes what it needs from the forward's inputs (it takes no out or logZ).
 * Every pass runs as dense tensor-core contractions over the virtual batch of the B*K
 * (sample, rank) pairs with the exponentials and rank reductions in element-wise kernels;
 * row maxima of A, B and x are taken out of every exponential (they cancel), so any
 * finite factors are in range. Precision: every contraction's products in the mode's
 * format (bf16 / TF32 / 3xTF32), float32 accumulation. flow_fp8 != 0 (the doc's opt-in
 * flow_precision "fp8"; precision auto only, ignored otherwise): the two flow
 * contractions (Fplus and Wstat) take e4m3 operands with a power-of-two scale per operand
 * row (largest magnitude within 448), float32 accumulation; the gradients and element
 * flows are not affected. The doc measures such statistics about 16x less accurate.
 * Limits: K >= 1, B <= 65535, B*K <= 2^22, M, N <= 2^24 (PC_ERR_SHAPE). M, N or B may
 * be 0. Workspace: pc_lowrank_sum_exp_workspace(..., with_backward, ...) bytes, 16-byte
 * aligned.
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_lowrank_sum_exp_workspace(int M, int N, int K, int B, int with_backward,
                                                   pc_precision_t prec, size_t* bytes);

PCSUM_API pc_status_t pc_lowrank_sum_exp_fwd(int M, int N, int K, int B, const float* theta,
                                             const float* A, const float* Bm, const float* x,
                                             float* out, float* logZ, pc_precision_t prec,
                                             void* ws, size_t ws_bytes, pc_stream_t stream);

PCSUM_API pc_status_t pc_lowrank_sum_exp_bwd(int M, int N, int K, int B, const float* theta,
                                             const float* A, const float* Bm, const float* x,
                                             const float* f, float* dA, float* dB, float* e,
                                             float* Fplus, float* Wstat, int accumulate, int flow_fp8,
                                             pc_precision_t prec, void* ws, size_t ws_bytes,
                                             pc_stream_t stream);

/* ------------------------------------------------------------------------------
 * HMM circuit with LowRank "exp_sum" transitions (pyjuice LowRank API doc: intro
 * formulas; Parameters: tie_external off, one pair of factor tensors per copy of the
 * tied transition node vector). The HMM of pc_hmm_fwd_bwd, except that the transition
 * layer of position t (t = 0 .. T-2) uses per-sample parameters
 *   A_b^(t)[k,l] = A[k,l] exp((FA[t][b] FB[t][b])[k,l]) / Z_b^(t)[k]
 * (Z normalizes each row over its children).
 *   tokens [B][T] int32, pi [H], A [H][H], E [H][V]      as for pc_hmm_fwd_bwd (device)
 *   FA [T-1][B][H][K], FB [T-1][B][K][H]                 the copies' factors, K <= 64
 *   ll [B] (double)                                      per-sample log-likelihood
 *   dpi [H], dE [H][V]                                   flows as for pc_hmm_fwd_bwd
 *   dA [H][H] = sum_t F+_t, Wstat [H][H] = sum_t W_t     the tied A's statistics (the
 *                                                        M-step's F+ and W, F- = A W)
 *   dFA, dFB (shaped as FA, FB)                          gradients of sum_b ll[b]
 * Each flow output may be NULL; with accumulate != 0 they are added to. Every transition
 * layer runs as pc_lowrank_exp_sum_fwd / _bwd (the scale is never stored); the results
 * are deterministic. Precision as for the LowRank layer. Errors: PC_ERR_SHAPE,
 * PC_ERR_UNSUPPORTED (K > 64), PC_ERR_NULL, PC_ERR_WORKSPACE, PC_ERR_ALIGNMENT.
 * Workspace: pc_hmm_lowrank_workspace bytes, 16-byte aligned.
 * ---------------------------------------------------------------------------- */
PCSUM_API pc_status_t pc_hmm_lowrank_workspace(int H, int T, int V, int B, int K, pc_precision_t prec,
                                               size_t* bytes);

PCSUM_API pc_status_t pc_hmm_lowrank_fwd_bwd(int H, int T, int V, int B, int K, const int32_t* tokens,
                                             const float* pi, const float* A, const float* E,
                                             const float* FA, const float* FB, double* ll, float* dpi,
                                             float* dA, float* Wstat, float* dE, float* dFA, float* dFB,
                                             int accumulate, pc_precision_t prec, void* ws,
                                             size_t ws_bytes, pc_stream_t stream);

/* ---------------------------------------------------------------- EM M-step
 * The M-step that follows the backward (pyjuice LowRank API doc, Training): for each of
 * the G*M nodes (rows), over its N children,
 *
 *   theta[g][i][j] = r[g][i][j] / sum_j' r[g][i][j'],
 *   r = F                          (W == NULL: the plain normalize(F) of the parameter
 *                                   flows of a sum layer, HMM or HCLT; Baum-Welch)
 *   r = F / W, 0 where W <= 0      (W != NULL: the LowRank conditional update
 *                                   normalize(theta * F+ / F-) with F- = theta * W)
 *
 * F, W, theta: device, row-major [G][M][N] float32, caller-owned; theta is read only
 * where a row's sum of r is zero or not finite (no flow reached the node): that row keeps
 * its parameters (the pages are silent there). Rows are independent; F and W are not
 * modified and may not alias theta. Asynchronous on `stream`, no workspace, capturable.
 * Errors: PC_ERR_NULL (F or theta NULL), PC_ERR_SHAPE (G, M, N < 1 or G*M >= 2^31);
 * nothing is launched then. */
PCSUM_API pc_status_t pc_em_normalize(int G, int M, int N, const float* F, const float* W, float* theta,
                                      pc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PCSUM_H_ */
