/*
 * gns.h — C ABI of libgns: batched Gram Newton-Schulz orthogonalization and the Muon step
 * around it, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes (the pages' definitions, restated):
 *   - Muon (Dion3: Full-Stack Orthogonal Updates, sec. 2.1 eq. (1)): M <- mu M + G;
 *     W <- W - eta * polar(M), polar(X) = U V^T from the SVD X = U S V^T (Definition 1).
 *   - polar is approximated by T odd-polynomial Newton-Schulz steps p_t(x) = a_t x + b_t x^3
 *     + c_t x^5 after Frobenius normalisation X <- X / (||X||_F + eps) (Dion3 sec. 2.2,
 *     Algorithm 1).
 *   - Gram Newton-Schulz (Dion3 sec. 4, Theorem 2, Algorithm 3) gets the same result from the
 *     n x n Gram matrix R = X X^T: Z_t = b_t R + c_t R^2, Q_t = Q_{t-1} Z_t + a_t Q_{t-1},
 *     RZ_t = R_{t-1} Z_t + a_t R_{t-1}, R_t = Z_t RZ_t + a_t RZ_t, with a restart
 *     (X <- Q X, R <- X X^T, Q <- I) after the iterations named in restart_mask; output Q_T X.
 *   - Symmetric products (Dion3 sec. 5): only upper-triangle tiles of a symmetric result are
 *     computed; each off-diagonal tile is also written to its mirrored position, diagonal
 *     tiles once.
 *   - Dion3 update rule (Dion3 sec. 6, Algorithm 4, Muon flavour): M <- M + G; S = the
 *     k = ceil(f n) rows of largest l1 norm; W <- (1 - eta wd) W; W[S] -= eta polar(M[S]);
 *     M[S] <- mu M[S].
 *   - NorMuon (Dion3 sec. 2.1 eq. (2) and the NorMuon steps of Algorithm 4): a per-row second moment
 *     v_i <- beta2 v_i + (1 - beta2) mean_j O_ij^2 of the orthogonalized update, rows divided
 *     by sqrt(v_i) + eps, the result rescaled to the Frobenius norm of O; fp32 arithmetic.
 *   - RowNorm and Periodic Row-wise Muon (Scaling Muon for Diffusion Transformers, sec. 3.1
 *     eq. (5), sec. 3.2 eq. (7)): R_eps(X)_i = X_i / max(||X_i||_2, eps) on the oriented
 *     momentum, scaled by gamma, used on the steps t with t mod K != 0; Newton-Schulz on the
 *     others.
 *   - Safety factor (Dion3 appendix B.2.2): every polynomial replaced by p_t(x / s), i.e.
 *     (a, b, c) -> (a / s, b / s^3, c / s^5).
 *
 * Conventions shared by every entry point:
 *   Matrices. A gns_batch describes `count` row-major matrices of one shape at a constant
 *     element stride (a "megabatch": Dion3 sec. 7 groups all same-shape matrices into one
 *     batch). All pointers are DEVICE addresses owned by the caller; the library never
 *     allocates or frees device memory. ptr must be 16-byte aligned; ld and stride must be
 *     multiples of 8 elements (16 bytes) for bf16 / fp16 and of 4 elements for fp32; ld >= cols,
 *     stride >= rows * ld (stride is ignored when count == 1). count and min(rows, cols) are
 *     at most 65535 and max(rows, cols) at most 4194240 (65535 x 64), the kernels' grid
 *     limits; larger values are argument errors.
 *   Orientation. A matrix with rows > cols is orthogonalized through its transpose and the
 *     result is mapped back (Dion3 Algorithm 1 assumes n <= m); no transposed copy is made.
 *   Streams. Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and returns without synchronising the host. The enqueued work is kernels and memsets
 *     only (a GEMM launch that follows the library's own norm pass may be a programmatic
 *     dependent launch: it starts its setup early and waits on the device for that pass),
 *     so a call may be recorded by stream capture into a CUDA graph and replayed; make
 *     one call on the device outside capture first (it looks up and caches the device's
 *     launch limits and the driver's tensor-map encoder).
 *   Workspace. Calls that need scratch take a caller-owned device buffer `ws` of at least
 *     gns_workspace_size(...) bytes (256-byte aligned).
 *   Errors. Argument errors are detected on the host and returned (nothing is enqueued).
 *     Conditions found on the GPU (non-finite outputs, a wait that timed out) are OR-ed
 *     into the optional device int32 *dev_status (bit 0: non-finite, bit 1: timeout); the
 *     caller reads it after synchronising. gns_last_error() gives a thread-local message.
 *   Aliasing. Outputs may not alias inputs unless stated.
 */
#ifndef GNS_H_
#define GNS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GNS_API __attribute__((visibility("default")))
#else
#define GNS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define GNS_VERSION 1
#define GNS_MAX_T 16

typedef enum {
  GNS_OK = 0,
  GNS_ERR_INVALID = -1,     /* bad argument (shape, alignment, null pointer, T range ...) */
  GNS_ERR_UNSUPPORTED = -2, /* valid request the library does not implement */
  GNS_ERR_WORKSPACE = -3,   /* ws too small or misaligned */
  GNS_ERR_CUDA = -4         /* a CUDA runtime call failed (launch, tensor-map encode ...) */
} gns_status;

/* device status bits (written by kernels, read by the caller after a sync) */
#define GNS_DEVST_NONFINITE 1
#define GNS_DEVST_TIMEOUT 2

typedef enum {
  GNS_BF16 = 0, /* bf16 storage, tensor-core products with fp32 accumulation (hot path) */
  GNS_F32 = 1,  /* fp32 storage and fp32 arithmetic (validation path) */
  GNS_F16 = 2   /* fp16 storage, tensor-core products with fp32 accumulation (Dion3 Algorithm 3
                   casts to float16; appendix B.2.2 prefers it to bfloat16) */
} gns_dtype;

/* `count` row-major matrices: element (b, i, j) at ptr + b*stride + i*ld + j (elements). */
typedef struct {
  void* ptr;
  int64_t count;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  int64_t stride;
} gns_batch;

/* Newton-Schulz schedule: T iterations with coefficients (a_t, b_t, c_t), t = 1..T
 * (index t-1), e.g. a caller's Polar Express table. Bit i of restart_mask (1 <= i < T)
 * restarts after iteration i (Dion3 Algorithm 3 restarts after iteration 2: mask 1u << 2).
 * eps as in the normalisation step of Algorithm 1. safety = s > 0 applies the safety factor of Dion3 appendix
 * B.2.2 to every iteration: p_t(x) becomes p_t(x / s), so (a, b, c) is used as
 * (a / s, b / s^3, c / s^5); s = 1 leaves the table as given (the pages' conservative choice
 * for Polar Express coefficients is s = 1.05). */
typedef struct {
  int32_t T;
  float a[GNS_MAX_T];
  float b[GNS_MAX_T];
  float c[GNS_MAX_T];
  uint32_t restart_mask;
  float eps;
  float safety;
} gns_ns_params;

/* Update flavours of gns_muon_step. */
typedef enum {
  GNS_FLAVOR_MUON = 0,     /* O = polar(M) (Dion3 eq. (1); Algorithm 4 Muon flavour) */
  GNS_FLAVOR_NORMUON = 1,  /* O = NorMuon-normalised polar(M) (Dion3 eq. (2); NorMuon steps of Algorithm 4) */
  GNS_FLAVOR_ROWNORM = 2,  /* O = gamma R_eps(M) (Scaling Muon for DiTs eq. (5)); dense only */
  GNS_FLAVOR_PERIODIC = 3  /* Periodic Row-wise Muon (ibid. eq. (7)): MUON when step % period
                              == 0, else ROWNORM; dense only */
} gns_flavor;

/* Muon step hyper-parameters. frac = 1: dense step; 0 < frac < 1: Dion3 fractional update
 * (Algorithm 4) with k = ceil(frac * n) selected rows. The weight update is
 * W <- (1 - lr*weight_decay) W - lr*scale*O, fp32 arithmetic and one bf16 rounding.
 * Fields after `frac` may be left zero: flavour MUON, Newton-Schulz in bf16.
 *   flavor        gns_flavor.
 *   ns_dtype      GNS_BF16 or GNS_F16: storage type of the Newton-Schulz products (W, G, M
 *                 stay bf16; with GNS_F16 the normalised momentum is rounded to fp16 once,
 *                 as in Dion3 Algorithm 3).
 *   beta2         NorMuon second-moment decay, in [0, 1).
 *   norm_eps      NorMuon: added to sqrt(v_i) (> 0). RowNorm: lower bound of a row norm
 *                 (> 0).
 *   rownorm_gamma RowNorm multiplier gamma (> 0; the page uses 0.15).
 *   period, step  Periodic Row-wise Muon: K >= 1 (the page uses 3) and the step index t. */
typedef struct {
  float lr;
  float momentum;
  float weight_decay;
  float scale;
  float frac;
  int32_t flavor;
  int32_t ns_dtype;
  float beta2;
  float norm_eps;
  float rownorm_gamma;
  int32_t period;
  int32_t step;
} gns_muon_params;

typedef enum {
  GNS_OP_GRAM_NS = 0,     /* gns_gram_ns_batched */
  GNS_OP_NS_STANDARD = 1, /* gns_ns_standard_batched */
  GNS_OP_MUON_STEP = 2,   /* gns_muon_step (dense or fractional per muon_params) */
  GNS_OP_FRAC_SELECT = 3  /* gns_frac_row_select */
} gns_op;

/* Library version (GNS_VERSION). */
GNS_API int gns_version(void);

/* Status name. */
GNS_API const char* gns_status_string(int status);

/* Copies the calling thread's last error message into buf (always NUL-terminated when
 * len > 0); returns its full length. */
GNS_API int gns_last_error(char* buf, size_t len);

/* Fills *p with the default schedule: T = 5, fixed quintic (a, b, c) = (3.4445, -4.7750,
 * 2.0315) every iteration (Scaling Muon for Diffusion Transformers, appendix D.3), restart
 * after iteration 2 (Dion3 Algorithm 3), eps = 1e-7 (the normalisation of Dion3 Algorithm 1), safety 1. */
GNS_API void gns_ns_params_default(gns_ns_params* p);

/* Bytes of workspace `op` needs for these batches (the same arguments as the call).
 * muon_params may be NULL except for GNS_OP_MUON_STEP / GNS_OP_FRAC_SELECT (frac, k).
 * Returns 0 and sets the last error on invalid arguments. */
GNS_API size_t gns_workspace_size(gns_op op, const gns_batch* x, int ngroups, gns_dtype dtype,
                          const gns_ns_params* ns, const gns_muon_params* muon);

/* Gram Newton-Schulz (Dion3 Algorithm 3 with the schedule in *ns) of every matrix of
 * ngroups batches x[g]; result written to out[g] (same shape and dtype as x[g]). A group
 * whose oriented shape is square (rows == cols) takes standard Newton-Schulz with
 * symmetric products instead, the alpha = 1 rule of Dion3 sec. 4.1 (same result in exact
 * arithmetic, fewer launches). out may not alias x. */
GNS_API int gns_gram_ns_batched(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                        const gns_ns_params* ns, void* ws, size_t ws_bytes, int32_t* dev_status,
                        void* stream);

/* Standard Newton-Schulz (Dion3 Algorithm 1, symmetric products for X X^T and A^2 as in
 * Dion3 sec. 2.3 / appendix C.3) with the same arguments. Restart bits are ignored. */
GNS_API int gns_ns_standard_batched(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                            const gns_ns_params* ns, void* ws, size_t ws_bytes, int32_t* dev_status,
                            void* stream);

/* Symmetric rank-K product (Dion3 sec. 5, the X X^T Gram product of Algorithm 3):
 * C <- alpha X X^T + beta C for every matrix of the batch; x is n x K, c is n x n; both
 * triangles of C are written (upper tiles computed, mirrored), diagonal tiles once.
 * beta != 0 reads C, which must then be symmetric. */
GNS_API int gns_sym_gemm_xxt(const gns_batch* x, const gns_batch* c, float alpha, float beta, gns_dtype dtype,
                     int32_t* dev_status, void* stream);

/* Symmetric product with addend (Dion3 sec. 5: "AB" and "alpha AB + beta C" assuming AB and
 * C symmetric): D <- alpha A B + beta C for n x n batches a, b, c, d (c may be NULL when
 * beta == 0; d may alias c; d may not alias a or b). Only upper tiles of A B are formed and
 * mirrored, so a non-symmetric A B yields its upper triangle reflected. */
GNS_API int gns_sym_gemm(const gns_batch* a, const gns_batch* b, const gns_batch* c, const gns_batch* d, float alpha,
                 float beta, gns_dtype dtype, int32_t* dev_status, void* stream);

/* One iteration of the loop of Dion3 Algorithm 3 (its Z, Q, RZ and R updates) on n x n batches, in place:
 *   Z  <- b R + c R^2
 *   Q  <- Q Z + a Q          (q_is_identity != 0: Q <- Z + a I without a product)
 *   RZ <- R Z + a R          (skipped when skip_r != 0)
 *   R  <- Z RZ + a RZ        (skipped when skip_r != 0)
 * Z and RZ are caller-provided scratch of the same shape; q_scratch (same shape) receives
 * Q_{t-1} Z + a Q_{t-1} before it is copied back into Q (it may be NULL when
 * q_is_identity != 0). */
GNS_API int gns_sym_poly_update(const gns_batch* R, const gns_batch* Q, const gns_batch* Z, const gns_batch* RZ,
                        const gns_batch* q_scratch, float a, float b, float c, int q_is_identity, int skip_r,
                        gns_dtype dtype, int32_t* dev_status, void* stream);

/* One optimizer step on ngroups bf16 batches (W, G, M of equal shapes per group):
 *   frac == 1: M <- mu M + G (fp32 arithmetic, bf16 store); O = Gram NS of M (oriented);
 *              W <- (1 - lr wd) W - lr scale O (in the final product's epilogue for the
 *              Muon flavour).
 *   frac <  1: Dion3 Algorithm 4: M <- M + G; S = top-k rows (columns when rows > cols) by
 *              exact l1 norm, ties to the lower index; O = Gram NS of M[S]; W <- (1 - lr wd) W;
 *              W[S] -= lr scale O; M[S] <- mu M[S].
 * Flavours (muon->flavor): NORMUON replaces O by the NorMuon update (eq. (2)) with the
 * second moments of the oriented rows in V; ROWNORM (and PERIODIC off its refresh steps)
 * replaces the Newton-Schulz of the dense step by O = gamma R_eps(M) of the oriented M.
 * V: NULL unless the flavour is NORMUON; then per group an fp32 batch of count x 1 x n,
 * n = min(rows, cols) (ld >= n, a multiple of 4), updated in place (row i of the oriented M;
 * for frac < 1 only the selected rows). W, G, M, V may not alias. */
GNS_API int gns_muon_step(const gns_batch* W, const gns_batch* G, const gns_batch* M, const gns_batch* V,
                  int ngroups, const gns_muon_params* muon, const gns_ns_params* ns, void* ws,
                  size_t ws_bytes, int32_t* dev_status, void* stream);

/* Selection step of Dion3 Algorithm 4 for one bf16 batch m: per matrix, the
 * k rows (columns when rows > cols) of largest exact l1 norm, ties to the lower index,
 * written ascending to idx[b*k .. b*k+k-1] (device int32). When gathered != NULL it also
 * receives the selected rows (count x k x cols, or k x rows for a tall matrix, i.e. the
 * selected rows of the oriented matrix). */
GNS_API int gns_frac_row_select(const gns_batch* m, int k, int32_t* idx, const gns_batch* gathered, void* ws,
                        size_t ws_bytes, void* stream);

/* Self-test of the failure detection every kernel of the library relies on (no GPU fault is
 * involved). Launches one thread that waits, through the same bounded-wait code the GEMM
 * kernel uses, first until the device int32 *counter reaches target (the cross-CTA completion
 * counters of a persistent launch) and then on an mbarrier phase that nothing completes (the
 * operand, accumulator and C rings), each wait giving up after limit_us microseconds
 * (1 .. 2000000; the library's own waits give up after 2 s). A wait that runs out ORs
 * GNS_DEVST_TIMEOUT into *dev_status (nullable) and the kernel returns normally, so the
 * context stays usable. out (nullable, device, two uint64): out[0] = nanoseconds spent in
 * both waits, out[1] = bit 0 set if the counter wait succeeded, bit 1 if the mbarrier wait
 * did (it cannot). The caller owns every buffer; argument errors return GNS_ERR_INVALID. */
GNS_API int gns_selftest_bounded_wait(const int32_t* counter, int32_t target, uint32_t limit_us,
                                      int32_t* dev_status, uint64_t* out, void* stream);

/* Size of the fixed scratch array behind gns_gram_ns_batched_noalloc (64 MiB). */
#define GNS_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* Same computation and arguments as gns_gram_ns_batched, minus the workspace, for callers
 * that cannot allocate device memory where they orthogonalize (a framework memory pool that
 * forbids allocations it does not own, a real-time loop that must not allocate after
 * start-up, a plug-in handed device pointers but no allocator). The scratch comes from a
 * fixed device array of GNS_NOALLOC_SCRATCH_BYTES compiled into the library, which every
 * GPU that loads the library's code reserves until the process exits; this call allocates
 * nothing. The pages have no counterpart of this entry point.
 * Returns GNS_ERR_WORKSPACE, with the reason in gns_last_error(), when the batches need more
 * scratch than that (gns_workspace_size(GNS_OP_GRAM_NS, ...) tells how much).
 * Every call outside stream capture looks up the array's device address with the call's
 * device current (so the address stays valid after a cudaDeviceReset); a call under capture
 * uses the address the last uncaptured call on that device found, so make the first call on
 * a device before any stream capture (a first call under capture returns GNS_ERR_INVALID).
 * All calls share the array: each call
 * resets the counters that must start at zero and writes every other scratch value before
 * reading it, and calls whose executions overlap on the GPU race on it — serialise them. */
GNS_API int gns_gram_ns_batched_noalloc(const gns_batch* x, const gns_batch* out, int ngroups, gns_dtype dtype,
                                        const gns_ns_params* ns, int32_t* dev_status, void* stream);

/* Optional instrumentation, off by default, per calling host thread.
 * gns_profile_set(events, capacity): events points to 2*capacity cudaEvent_t handles the
 * caller created; from now on every tensor-core / fp32 GEMM launch the library enqueues is
 * bracketed by cudaEventRecord(events[2i]) and cudaEventRecord(events[2i+1]) on the launch
 * stream (i counts launches; launches beyond capacity are not recorded), and the counters
 * below restart from zero. events == NULL switches recording off (counting goes on).
 * gns_profile_query(&gemm_launches, &all_launches): GEMM launches and kernel launches of
 * any kind (memsets excluded) enqueued since the last gns_profile_set on this thread. */
GNS_API int gns_profile_set(void** events, int capacity);
GNS_API int gns_profile_query(int* gemm_launches, int* all_launches);

#ifdef __cplusplus
}
#endif

#endif /* GNS_H_ */
