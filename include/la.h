/*
 * la.h - C ABI of a GB300 (sm_103a) library for kernelised linear attention
 * with the feature map phi(x) = elu(x) + 1.
 *
 * Method: "Transformers are RNNs: Fast Autoregressive Transformers with Linear
 * Attention" (Katharopoulos et al.), read in its Chinese translation.  Per
 * head, with Q, K in R^{N x D} and V in R^{N x M} (sec. 3.1 and 3.2.1
 * notation; rows are positions):
 *
 *   phi(x)       = x + 1 (x > 0), exp(x) (x <= 0)            sec. 3.2.1 eq. (7)
 *   non-causal   V'_i = phi(Q_i)^T (sum_j phi(K_j) V_j^T)
 *                       / phi(Q_i)^T (sum_j phi(K_j))          sec. 3.2 eq. (5)
 *   causal       the same sums over j <= i:                   sec. 3.3 eq. (9)
 *                S_i = S_{i-1} + phi(K_i) V_i^T,  Z_i = Z_{i-1} + phi(K_i),
 *                V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i        eqs. (10)-(12)
 *   decode       one step of eqs. (18)-(20): update s, z, then read out
 *                (the layer's f_l and residual are not part of this library).
 *
 * There is no epsilon in any denominator and no 1/sqrt(D) inside phi: phi > 0,
 * so every denominator is a sum of positive terms.
 *
 * Conventions for every entry point
 * ---------------------------------
 * Layout:    contiguous row-major.  Q, K: [B, H, N, D]; V, out: [B, H, N, M];
 *            state S: [B, H, D, M] fp32 (S[d][m] = sum phi(K)_d V_m);
 *            z: [B, H, D] fp32.  Decode q, k: [B, H, D]; v, y: [B, H, M].
 * Types:     Q, K, V and out share one dtype (LA_DTYPE_F32 or LA_DTYPE_BF16);
 *            all arithmetic is fp32 (bf16 operands on tensor cores accumulate
 *            in fp32); the state is always fp32; bf16 results are rounded to
 *            nearest-even once.
 * Sizes:     D, M in {16, 32, 64, 128}; B, H, N >= 0.  An empty problem
 *            (B*H*N == 0) is valid and launches nothing.
 * Pointers:  device pointers (or pointers the GPU can dereference), 16-byte
 *            aligned.  The caller owns every buffer, the workspace and the
 *            stream; the library allocates no device memory and keeps no
 *            state besides cached device properties and a per-device error
 *            word.  Inputs are read-only; out must not alias an input.
 * Stream:    a cudaStream_t (NULL = legacy default stream).  Work is enqueued
 *            asynchronously; the call returns once it is enqueued.
 * Errors:    argument checks happen on the host before any launch and return
 *            LA_ERR_INVALID_ARG (bad pointer, alignment, negative size,
 *            workspace too small) or LA_ERR_UNSUPPORTED (D or M outside the
 *            supported set).  A failed launch returns LA_ERR_CUDA.  A kernel
 *            that gives up waiting (every wait in the library is bounded)
 *            records LA_ERR_TIMEOUT in the device error word, which
 *            la_get_last_error() reports.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,
    LA_ERR_UNSUPPORTED = 2,
    LA_ERR_CUDA = 3,
    LA_ERR_TIMEOUT = 4,
    LA_ERR_BOUNDS = 5      /* checked build only: an access outside a buffer was caught and skipped */
} la_status;

typedef enum { LA_DTYPE_F32 = 0, LA_DTYPE_BF16 = 1 } la_dtype;

typedef enum {
    LA_OP_NONCAUSAL = 0,
    LA_OP_CAUSAL = 1,
    LA_OP_DECODE = 2,
    LA_OP_NONCAUSAL_BWD = 3,
    LA_OP_CAUSAL_BWD = 4
} la_op;

typedef struct {
    int B, H, N, D, M;
    la_dtype dtype;
} la_shape;

/*
 * Bytes of device workspace the call `op` needs for shape `s` and chunk
 * length `chunk` (0 = default).  0 means the call needs none and accepts a
 * NULL workspace.  Returns (size_t)-1 for an invalid shape.
 */
size_t la_workspace_bytes(la_op op, la_shape s, int chunk);

/*
 * Non-causal attention, sec. 3.2 eq. (5): the summaries sum_j phi(K_j) V_j^T
 * (D x M) and sum_j phi(K_j) (D) are reduced once per head over all N keys in
 * fp32, then every query row reads them out.
 *   q, k: [B,H,N,D]; v: [B,H,N,M]; out: [B,H,N,M] (same dtype as q).
 *   workspace: la_workspace_bytes(LA_OP_NONCAUSAL, s, 0) bytes, device memory.
 */
la_status la_forward_noncausal(const void *q, const void *k, const void *v, void *out,
                               la_shape s, void *workspace, size_t ws_bytes,
                               la_stream_t stream);

/*
 * Causal attention, sec. 3.3 eqs. (9)-(12), computed chunk by chunk: within a
 * chunk of rows the masked products phi(Q) phi(K)^T (j <= i, the diagonal
 * kept) multiply V; the rows see earlier chunks through the carried fp32
 * state (S, z).  This regrouping of the sums of eq. (9) is exact in real
 * arithmetic; results for different chunk lengths differ only by rounding.
 *   out: [B,H,N,M] or NULL (state only, e.g. to prefill a decoder).
 *   chunk: 0 (library default), 64 or 128 (anything else is
 *      LA_ERR_UNSUPPORTED).  It is a hint, not a contract: the bf16
 *      tensor-core path (D, M in {64, 128}) always groups 128 rows, one
 *      tcgen05 M = 128 tile per chunk, and the CUDA-core path (fp32, other
 *      D, M) always groups 32 rows; every accepted value gives the same
 *      result up to rounding.
 *   S: [B,H,D,M] fp32, z: [B,H,D] fp32: both NULL (start from s_0 = 0, z_0 = 0,
 *      eqs. (16)-(17)) or both non-NULL: the call starts from the state they
 *      hold and overwrites them with the state after the last token.  Exactly
 *      one NULL is LA_ERR_INVALID_ARG.
 *   workspace: la_workspace_bytes(LA_OP_CAUSAL, s, chunk) bytes.
 */
la_status la_forward_causal(const void *q, const void *k, const void *v, void *out,
                            la_shape s, int chunk, float *S, float *z,
                            void *workspace, size_t ws_bytes, la_stream_t stream);

/*
 * One recurrent step, sec. 3.4 eqs. (18)-(20), for B*H independent heads:
 *   S <- S + phi(k) v^T,  z <- z + phi(k),  y = phi(q)^T S / phi(q)^T z
 * (state updated first, then read out).  s.N is ignored.
 *   q, k: [B,H,D]; v, y: [B,H,M] (dtype s.dtype); S, z fp32 updated in place.
 */
la_status la_decode_step(const void *q, const void *k, const void *v, void *y,
                         float *S, float *z, la_shape s, la_stream_t stream);

/*
 * Causal attention over a batch of sequences of different lengths (a prefill
 * of several prompts at once): as la_forward_causal, but batch entry b has
 * lens[b] tokens (clamped to [0, N]); rows at or past its length are read but
 * add nothing, and their rows of `out` are unspecified.  With S, z the call
 * starts each head from its state and leaves the state after its own length
 * (a zero length leaves it unchanged).
 *   lens: device pointer to B int32 lengths (4-byte aligned).
 *   q, k, v, out, S, z, workspace: as la_forward_causal (chunk = 0).
 */
la_status la_forward_causal_varlen(const void *q, const void *k, const void *v, void *out, const int *lens,
                                   la_shape s, float *S, float *z, void *workspace, size_t ws_bytes,
                                   la_stream_t stream);

/*
 * T recurrent steps, sec. 3.4 eqs. (18)-(20), in one launch: each head's state
 * is read once, updated and read out T times on chip, and written back once.
 * Step-major inputs: q, k [T,B,H,D]; v, y [T,B,H,M]; S, z as la_decode_step.
 * For when several steps' inputs are known together (a verified draft, a
 * teacher-forced continuation): the result equals T calls of la_decode_step,
 * which is the causal form over those T tokens started from (S, z); for bf16
 * with D, M in {64, 128} it runs the chunked tensor-core causal kernel.
 *   steps: device pointer to B int32 step counts (clamped to [0, T]; batch
 *      entry b runs its first steps[b] steps; its later y rows are
 *      unspecified), or NULL for all T.  s.N is ignored.
 */
la_status la_decode_steps(const void *q, const void *k, const void *v, void *y, float *S, float *z,
                          const int *steps, int T, la_shape s, la_stream_t stream);

/*
 * Backward of the causal form (the gradient sec. 3.3.1 computes as cumulative
 * sums in constant extra memory; its eqs. (13)-(15) are not printed on the
 * page, so this is the chain rule through eqs. (10)-(12)).  Given
 * dout = dL/dV' it writes dq, dk, dv = dL/dQ, dL/dK, dL/dV:
 *   g_i = dout_i / den_i,  e_i = -(g_i . num_i) / den_i,
 *   dphi(Q_i) = S_i g_i + e_i Z_i                       (forward sweep)
 *   R_i = sum_{j>=i} phi(Q_j) g_j^T,  r_i = sum_{j>=i} e_j phi(Q_j)
 *   dphi(K_i) = R_i V_i + r_i,  dV_i = R_i^T phi(K_i)    (reverse sweep)
 * and dQ = dphi(Q) phi'(Q), dK = dphi(K) phi'(K), phi'(x) = 1 (x > 0), e^x.
 *   q, k, dq, dk: [B,H,N,D]; v, dout, dv: [B,H,N,M], all of dtype s.dtype;
 *   the gradients may not alias the inputs or each other.
 *   S0, z0: [B,H,D,M], [B,H,D] fp32, the state the forward started from
 *      (both NULL: zero); dSN, dzN: gradient reaching the forward's final
 *      state (both NULL: zero); dS0, dz0: receive dL/dS_0, dL/dZ_0 (both NULL:
 *      not wanted).  Chaining the backward of consecutive segments through
 *      dS0 -> dSN reproduces the backward of the whole sequence.
 *   workspace: la_workspace_bytes(LA_OP_CAUSAL_BWD, s, 0) bytes: g and e of
 *      every token, and (segmented route) the fp32 sums [S | Z] and [R | r]
 *      entering and leaving every segment, D*M + D floats each.
 * bf16 runs on tensor cores (tcgen05: bf16 operands, the state and the
 * reverse sums entering the products as bf16 hi + lo pairs, fp32
 * accumulation): with D = M = 64 in two sweeps of one CTA per head; with
 * D, M in {64, 128} otherwise in segments of consecutive 128-row chunks,
 * about one CTA per SM, the state held in TMEM along each segment (segment
 * key sums, a scan, a query pass, the reverse scan, a key pass).  fp32, and
 * bf16 at other sizes, run fp32 arithmetic on CUDA cores.  Errors as
 * la_forward_causal.
 */
la_status la_backward_causal(const void *q, const void *k, const void *v, const void *dout,
                             void *dq, void *dk, void *dv, la_shape s,
                             const float *S0, const float *z0, const float *dSN, const float *dzN,
                             float *dS0, float *dz0, void *workspace, size_t ws_bytes,
                             la_stream_t stream);

/*
 * Backward of the non-causal form, sec. 3.2 eq. (5): the same steps with the
 * sums over all N keys (S, Z the full sums, R and r summed over all queries).
 *   Arguments as la_backward_causal without the state ones;
 *   workspace: la_workspace_bytes(LA_OP_NONCAUSAL_BWD, s, 0) bytes (fp32
 *      partial sums of S, Z and of R, r per key or query range).
 * bf16 with D, M in {64, 128} runs on tensor cores in three launches (key
 * sums; a query pass giving dQ and the partial R, r; a key pass giving dK,
 * dV), the sums entering the products as bf16 hi + lo pairs; every other
 * dtype and size runs fp32 arithmetic on CUDA cores.
 */
la_status la_backward_noncausal(const void *q, const void *k, const void *v, const void *dout,
                                void *dq, void *dk, void *dv, la_shape s,
                                void *workspace, size_t ws_bytes, la_stream_t stream);

/* ------------------------------------------------------------------ variants
 * Other feature maps, read-out normalisations and the delta update rule.
 * Sources: "Transformers are RNNs" (TaR) sec. 3.2.1 (the degree-2 polynomial
 * kernel and its exact feature map) and "Linear Transformers Are Secretly
 * Fast Weight Programmers" (FWP: the DPFP feature map, sum normalisation, the
 * delta update rule), whose summary page lost its equations; each rule below
 * is the plainest reading of its prose.
 *
 * Feature map phi: R^D -> R^F, applied to every row of Q and K:
 *   LA_FM_ELU1   elu(x) + 1 (TaR eq. (7)); F = D.
 *   LA_FM_DPFP   DPFP-nu (FWP): r = [relu(x), relu(-x)] in R^{2D}; feature
 *                (s-1)*2D + i is r_i * r_{(i+s) mod 2D} for s = 1..nu,
 *                i = 0..2D-1; F = 2*D*nu, 1 <= nu < 2D.
 *   LA_FM_POLY2  degree-2 polynomial kernel (q.k)^2 (TaR sec. 3.2.1):
 *                feature a*D + b is x_a x_b; F = D^2.
 * Read-out (norm):
 *   LA_NORM_DEN  y_i = phi(q_i)^T S_i / phi(q_i)^T z_i, z_i = sum phi(k_j)
 *                (TaR eq. (12); FWP's "accumulator").
 *   LA_NORM_SUM  phi(q) and phi(k) are divided by the sum of their
 *                components (FWP); y_i = phi(q_i)^T S_i, no denominator.
 *   LA_NORM_NONE y_i = phi(q_i)^T S_i.
 * Update of the state S (F x M):
 *   LA_UPDATE_SUM    S_i = S_{i-1} + phi(k_i) v_i^T (TaR eq. (10)).
 *   LA_UPDATE_DELTA  vbar_i = S_{i-1}^T phi(k_i) (the value now paired with
 *                    k_i); S_i = S_{i-1} + phi(k_i) (beta_i (v_i - vbar_i))^T,
 *                    which stores beta_i v_i + (1 - beta_i) vbar_i in its place
 *                    (FWP); beta_i in [0, 1] is an input per token and head.
 * The read-out of token i follows its update (TaR eqs. (18)-(20)).
 * Supported: F <= 512; DPFP with LA_NORM_SUM or LA_NORM_NONE (with the
 * denominator, a query whose adjacent sign pairs match no earlier key gets
 * 0/0); POLY2 with LA_NORM_DEN or LA_NORM_NONE (its features can be
 * negative); LA_UPDATE_DELTA with LA_NORM_SUM only (|phi(k)|^2 <= 1 keeps
 * the state bounded).  Other combinations return LA_ERR_UNSUPPORTED;
 * unknown enum values LA_ERR_INVALID_ARG.
 * State layout: S [B, H, F, M] fp32 (S[f][m]); z [B, H, F] fp32 (LA_NORM_DEN
 * only).  Arithmetic: bf16 inputs of a sum-update variant with F, M in
 * {64, 128} (elu + 1 raw, sum-normalised or with the denominator; DPFP from
 * D = 64 / nu = 1, D = 32 / nu = 1 or 2, D = 16 / nu = 2 or 4), and of
 * the delta rule with sum-normalised features of width 64 (elu + 1 at
 * D = 64, DPFP at D = 32 / nu = 1 or D = 16 / nu = 2) and M = 64, run on
 * tensor cores (bf16 feature rows and operands, fp32 accumulation and
 * state; the delta rule's triangular solve in fp32 on CUDA cores); every
 * other case runs fp32 arithmetic on CUDA cores.
 */
typedef enum { LA_FM_ELU1 = 0, LA_FM_DPFP = 1, LA_FM_POLY2 = 2 } la_feature_map;
typedef enum { LA_NORM_DEN = 0, LA_NORM_SUM = 1, LA_NORM_NONE = 2 } la_norm;
typedef enum { LA_UPDATE_SUM = 0, LA_UPDATE_DELTA = 1 } la_update;

typedef struct {
    la_feature_map feature_map;
    int nu;                 /* DPFP shifts (ignored by the other maps) */
    la_norm norm;
    la_update update;
} la_variant;

/* F, the width of phi(x) for x in R^D under `var`; 0 if `var` is invalid. */
int la_feature_dim(la_variant var, int D);

/*
 * Bytes of device workspace la_forward_noncausal_variant needs (0 for the
 * causal and decode calls, which need none); (size_t)-1 if invalid.
 */
size_t la_variant_workspace_bytes(la_op op, la_shape s, la_variant var);

/*
 * Causal form of a variant over [B,H,N,.] inputs:
 *   q, k: [B,H,N,D]; v, out: [B,H,N,M]; beta: [B,H,N] (LA_UPDATE_DELTA,
 *      else ignored and may be NULL); all of dtype s.dtype.
 *   out may be NULL (state only).
 *   S: [B,H,F,M] fp32 or NULL; z: [B,H,F] fp32 or NULL.  With LA_NORM_DEN
 *      both or neither (as la_forward_causal); otherwise z must be NULL.  A
 *      given state is the starting state and receives the final state.
 * Errors as la_forward_causal.
 */
la_status la_forward_causal_variant(const void *q, const void *k, const void *v, const void *beta,
                                    void *out, la_shape s, la_variant var, float *S, float *z,
                                    la_stream_t stream);

/*
 * Non-causal form of a variant (LA_UPDATE_SUM only): KV = sum_j phi(K_j) V_j^T
 * and, for LA_NORM_DEN, sum_j phi(K_j) over all N keys, then y_i =
 * phi(Q_i)^T KV (/ phi(Q_i)^T sum_j phi(K_j)).
 *   workspace: la_variant_workspace_bytes(LA_OP_NONCAUSAL, s, var) bytes.
 */
la_status la_forward_noncausal_variant(const void *q, const void *k, const void *v, void *out,
                                       la_shape s, la_variant var, void *workspace, size_t ws_bytes,
                                       la_stream_t stream);

/*
 * One recurrent step of a variant: q, k [B,H,D]; v, y [B,H,M]; beta [B,H]
 * (delta rule); S [B,H,F,M] and (LA_NORM_DEN) z [B,H,F] fp32 updated in
 * place; z must be NULL otherwise.  s.N is ignored.
 */
la_status la_decode_step_variant(const void *q, const void *k, const void *v, const void *beta, void *y,
                                 float *S, float *z, la_shape s, la_variant var, la_stream_t stream);

/*
 * Non-causal attention that allocates nothing, for callers that cannot
 * allocate device memory: code that only receives pointers from a host
 * framework owning the device memory pool, or a loop that must not call the
 * allocator once it is running (cudaMalloc and cudaFree synchronise the
 * device).  No counterpart in the paper: it computes what
 * la_forward_noncausal computes (on the CUDA-core kernels, with the number of
 * key splits capped so that the partial sums fit), but its fp32 partial sums
 * live in an 8 MiB array compiled into this library (a file-scope __device__
 * array, held by every GPU that loads the library until the process exits)
 * instead of a caller workspace.
 *   Limit: B*H*(D*M + D)*4 bytes must not exceed 8 MiB (for D = M = 64,
 *   B*H <= 504; for D = M = 128, B*H <= 127); larger problems return
 *   LA_ERR_UNSUPPORTED before any launch.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Every call shares the one array: calls that overlap on the GPU (on two
 *   streams, or from two threads) race and corrupt each other's results.  The
 *   array keeps the last call's contents; nothing in it needs to start at
 *   zero (each call overwrites every partial sum it reads).
 * Arguments, layout and errors as la_forward_noncausal.
 */
la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v, void *out,
                                       la_shape s, la_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's error
 * word (LA_ERR_TIMEOUT if a kernel gave up a bounded wait since the last call)
 * or LA_ERR_CUDA if the stream itself reports an error.
 */
la_status la_get_last_error(la_stream_t stream);

/* Static English name of a status code. */
const char *la_status_string(la_status st);

/* Library version as major * 10000 + minor * 100 + patch. */
int la_version(void);

/*
 * Number of kernels this process has launched through the library so far
 * (all devices).  Benchmarks read it before and after a timed region.
 */
unsigned long long la_launch_count(void);

/*
 * 1 if this library is the checked build (liblinattn_checked.so, compiled
 * with -DLA_CHECKED), 0 for the release build (liblinattn.so).  The checked
 * build has no counterpart in the method: it is the release kernels with a
 * bounds check in front of each global-memory access whose index is computed
 * from run-time values other than the launch grid -- in the causal
 * tensor-core kernel the per-sequence length read, the carried-in state and
 * segment-workspace loads, the final-state stores and the direct output-row
 * stores; in the segment-sum pre-pass its workspace slot writes; in the
 * non-causal tensor-core kernel (exchange through the workspace) and in the
 * non-causal CUDA-core kernels (also used by la_forward_noncausal_noalloc)
 * the workspace slot writes and reads; in the non-causal tensor-core backward
 * the reads and writes of its partial sums.  TMA copies are clipped to their tensor
 * maps by the hardware, and the decode kernels index by block and thread
 * alone, so neither carries a check.  A failed check skips its access and
 * records LA_ERR_BOUNDS in the device error word, which la_get_last_error()
 * reports; nothing traps.  Results are otherwise identical to the release
 * build's; it is slower and meant for testing.
 */
int la_checked_build(void);

/*
 * Test hook of the checked build (a no-op in the release build): while
 * `enable` is non-zero, launches made by this process index past a buffer on
 * purpose, where the check catches it: the causal tensor-core kernel offsets
 * the rows of its carried-in state loads by D, the segment-sum pre-pass and
 * the non-causal CUDA-core reduction offset their workspace slot by the
 * workspace's whole length.  The call then reports LA_ERR_BOUNDS, and no access left
 * its buffer.
 */
void la_debug_inject_bounds(int enable);

/*
 * Test hook (no counterpart in the method): when `enable` is non-zero, the
 * next causal tensor-core launches on this process wait on a flag that nothing
 * ever sets, with a wait limit of about `limit_us` microseconds, before they
 * touch any data; they then record LA_ERR_TIMEOUT, release their tensor memory
 * and return.  Exercises the bounded-wait error path without hanging a GPU.
 */
void la_debug_inject_timeout(int enable, int limit_us);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
