/*
 * gsi.h -- C ABI of the gated-subspace linear map on one sm_103a GPU.
 *
 * The method ("Gated Subspace Inference for Transformer Acceleration",
 * gist.science technical summary):
 *
 *   §2.1 core decomposition.  For a linear map W (d_out x d) and a token
 *        x (length d), with an orthonormal rank-k basis V_k (d x k):
 *        x = V_k V_k^T x + r,  y = W x = (W V_k)(V_k^T x) + W r = M g + W r,
 *        where M = W V_k is the cached low-rank weight image (d_out x k) and
 *        g = V_k^T x the projection (length k).
 *   §2.2 gated residual step.  Per token, rho = ||r|| / ||x||.  If rho < eps
 *        the token takes the fast path y = M g (reads M, k columns' worth,
 *        instead of W); if rho >= eps it takes the exact slow path y = W x.
 *        Theorem 4 bounds the fast-path error by ||W||_2 * eps * ||x||.
 *   §2.2 (all linear maps) / §3.  The gate applies to every projection of a
 *        transformer layer (QKV, output, MLP up, MLP down).
 *
 * Conventions shared by every entry point:
 *   - All matrices are dense and row-major.  X is T x d (token t is row t),
 *     W is d_out x d, V is d x k, M is d_out x k, Y is T x d_out (float32).
 *     flags is T bytes (1 = slow path, 0 = fast path); rho is T float32.
 *   - W, V, M and X share one element type (gsi_dtype).  Accumulation is
 *     always float32.  For GSI_BF16 the caller supplies the k x k float32
 *     Gram matrix V^T V (built by gsi_build_image): a bf16-rounded basis is
 *     not exactly orthonormal and the library evaluates ||x - V g||^2 as
 *     ||x||^2 - 2||g||^2 + g^T (V^T V) g, which is exact for any basis.
 *     For GSI_F32 the Gram may be NULL, meaning "V is orthonormal"
 *     (||r||^2 = ||x||^2 - ||g||^2).
 *   - Readings where the pages are silent: a tie rho == eps is slow; a zero
 *     token has rho = 0 (fast, y = 0); a token with a NaN/Inf has rho = NaN
 *     and is slow.  eps = +inf is allowed (static projection: all fast).
 *   - Pointers to matrices, vectors and the workspace are DEVICE pointers;
 *     the arrays of pointers passed to gsi_stack and the status outputs
 *     (bytes, counts) are HOST pointers.  The caller owns every buffer; the
 *     library allocates nothing in these calls.
 *   - Every device pointer must be 16-byte aligned, the workspace 256-byte
 *     aligned.  d * sizeof(elem) and k * sizeof(elem) must be multiples of
 *     16 bytes (d, k multiples of 8 for bf16, of 4 for f32); otherwise the
 *     call returns GSI_ERR_UNSUPPORTED.  k <= GSI_MAX_K and k <= d.
 *   - Execution is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Argument errors are reported synchronously,
 *     before anything is enqueued; launch failures return GSI_ERR_CUDA.
 *     Device-side faults surface on the caller's next synchronisation.
 *   - The gate's decision never leaves the device: no call synchronises the
 *     stream, so calls may be captured into a CUDA graph.
 *   - On any non-OK status, gsi_last_error() returns a message for the
 *     calling thread.
 */
#ifndef GSI_H
#define GSI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GSI_MAX_K 512

typedef enum gsi_status {
  GSI_OK = 0,
  GSI_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad eps, misalignment */
  GSI_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle     */
  GSI_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  GSI_ERR_WORKSPACE = 4,   /* workspace missing, too small or misaligned    */
  GSI_ERR_TIMEOUT = 5      /* a bounded device wait gave up (see gsi_workspace_status) */
} gsi_status;

typedef enum gsi_dtype { GSI_F32 = 0, GSI_BF16 = 1 } gsi_dtype;

/* Which kernels run the map.
 *   FUSED  -- one launch per call for T <= 2.  One token: the single-token
 *             decode kernel, in which each 16-CTA cluster holds all of V in
 *             shared memory (or, for wider bases, the clusters exchange
 *             slices of g through epoch-tagged words in the workspace) and
 *             every CTA decides and applies; two tokens: every cluster
 *             projects on its share of V, with a grid barrier on the
 *             workspace where V does not fit a cluster;
 *   STREAM -- two launches (projection kernel, then decide-and-apply), any T;
 *   TENSOR -- tcgen05 contractions, bf16 only, for prefill-sized T;
 *   BATCH  -- bf16 maps, 2 <= T <= 16: the small-batch decode kernel, one
 *             launch per call.  Every CTA projects its slab of V on all T
 *             tokens, the clusters exchange slices of G through epoch-tagged
 *             words in the workspace, every CTA takes the same flags, and the
 *             three products (X V, G M^T for the fast tokens, X W^T for the
 *             slow ones) run as warp-level tensor-core products (bf16
 *             operands, float32 accumulation; G enters M G as a high and a
 *             low bf16 part).  Needs k a multiple of 64 (at most 384), d a
 *             multiple of 8 and d_out / (grid size) at most 160 rows.
 * AUTO picks FUSED for T = 1, and for T = 2 on float32 maps, where a slab of
 * V fits shared memory (and STREAM at run time on a device that cannot hold
 * the fused grid); BATCH for bf16 maps with 2 <= T <= 16 where its plan
 * fits; TENSOR for bf16 maps with T >= 9 otherwise; STREAM otherwise.  BATCH
 * and FUSED fall back to those choices at run time where the device cannot
 * run them.  Where the fused kernels' CTAs
 * wait on other clusters, they are launched as a co-resident (cooperative)
 * grid: a grid that cannot be co-resident is refused at launch, and AUTO
 * then runs the call on the STREAM kernels.  GSI_COOPERATIVE=0 in the
 * environment launches them without the co-resident attribute (grid sized
 * from the occupancy query; for profilers that relaunch kernels without it).
 * Every device wait stays bounded (~2 s, then GSI_ERR_TIMEOUT from
 * gsi_workspace_status, after which the workspace must be re-initialised).
 * A cluster kernel that finds itself running without its cluster shape sets
 * bit 13 of the error word and returns without touching other CTAs. */
typedef enum gsi_path {
  GSI_PATH_AUTO = 0,
  GSI_PATH_STREAM = 1,
  GSI_PATH_TENSOR = 2,
  GSI_PATH_FUSED = 3,
  GSI_PATH_BATCH = 4
} gsi_path;

/* One linear map with its cached artefacts (all device pointers). */
typedef struct gsi_map_desc {
  int64_t d;        /* input dimension (columns of W, rows of V)      */
  int64_t d_out;    /* output dimension (rows of W and M)             */
  int64_t k;        /* subspace rank (columns of V and M)             */
  gsi_dtype dtype;  /* element type of W, V, M and of the tokens X    */
  const void* W;    /* d_out x d                                      */
  const void* V;    /* d x k, orthonormal columns (up to rounding)    */
  const void* M;    /* d_out x k, the image W V (from gsi_build_image)*/
  const float* gram;/* k x k float32 V^T V; required for GSI_BF16     */
} gsi_map_desc;

/* §2.1: build the cached low-rank weight image M = W V (float32 accumulate,
 * rounded to nearest-even into `dtype`) and, if `gram` is non-NULL, the
 * float32 Gram matrix V^T V.  One-off per map.  W: d_out x d, V: d x k,
 * M: d_out x k (output), gram: k x k float32 (output, nullable). */
gsi_status gsi_build_image(const void* W, const void* V, void* M, float* gram,
                           int64_t d, int64_t d_out, int64_t k, gsi_dtype dtype,
                           void* stream);

/* §2.1 image build on the tensor cores.  gsi_build_image_ex computes what
 * gsi_build_image does; for GSI_BF16 maps with a scratch area M runs on
 * tcgen05 (V^T formed in the scratch, then M = W V as a tensor-core
 * contraction with float32 accumulation in TMEM, rounded to nearest even
 * into bf16).  The Gram matrix stays on the CUDA cores (float32 FMA chains):
 * the gate's residual needs it to float32 accuracy.  work: device, 256-byte aligned, at least
 * gsi_build_image_work_bytes(d, k, dtype) bytes (0 for GSI_F32, which keeps
 * the CUDA-core kernel, as does work == NULL); its first 256 bytes hold an
 * error word that gsi_workspace_status reads (a bounded wait of the
 * contraction gave up).  Enqueued on `stream`; allocates nothing. */
size_t gsi_build_image_work_bytes(int64_t d, int64_t k, gsi_dtype dtype);
gsi_status gsi_build_image_ex(const void* W, const void* V, void* M, float* gram, int64_t d, int64_t d_out, int64_t k,
                              gsi_dtype dtype, void* work, size_t work_bytes, void* stream);

/* Bytes of device workspace gsi_linear needs for `map` and T tokens with the
 * given path (host-only arithmetic, no device call).  *bytes is a HOST
 * pointer. */
gsi_status gsi_linear_workspace_size(const gsi_map_desc* map, int64_t T, gsi_path path,
                                     size_t* bytes);

/* Zero a workspace before its first use (its control words must start at
 * zero; calls keep them consistent from then on, so it is zeroed once).
 * Zero it again after a call has reported GSI_ERR_TIMEOUT.  A workspace
 * serves one stream at a time.  Enqueued on `stream`. */
gsi_status gsi_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Read the device error word of a workspace (SYNCHRONISES `stream`).
 * *code = 0 when no bounded wait has given up since the last init. */
gsi_status gsi_workspace_status(const void* workspace, uint32_t* code, void* stream);

/* §2.1-§2.2 gate only: projections G (T x k float32), residual ratios rho
 * (T float32, nullable) and flags (T bytes) for T tokens X. */
gsi_status gsi_gate(const gsi_map_desc* map, const void* X, int64_t T, float eps,
                    float* G, float* rho, uint8_t* flags,
                    void* workspace, size_t ws_bytes, void* stream);

/* §2.1 core decomposition, checked (a validation mode, off the hot path).
 * The gate kernels evaluate ||x - V g||^2 from the Gram form without a
 * second pass over V.  This call forms the residual itself, r_t = x_t - V g_t,
 * for the projections G (T x k float32, as written by gsi_gate) with a second
 * pass over V, and writes rho_explicit[t] = ||r_t|| / ||x_t|| (T float32; 0
 * for a zero token) and *max_dev = max over tokens of
 * |rho[t]^2 - rho_explicit[t]^2| (one float32), rho (T float32) being the
 * gate's ratios; tokens where either value is not finite are skipped.
 * Partial sums in float32 per 64-row slab of V, added in slab order in
 * double: bitwise reproducible.  work: device, 256-byte aligned,
 * gsi_residual_check_work_bytes(d, T) bytes.  All array arguments are device
 * pointers; T <= 524280.  Enqueued on `stream`. */
size_t gsi_residual_check_work_bytes(int64_t d, int64_t T);
gsi_status gsi_residual_check(const gsi_map_desc* map, const void* X, int64_t T, const float* G, const float* rho,
                              float* rho_explicit, float* max_dev, void* work, size_t work_bytes, void* stream);

/* §2.2 per-token gate, compaction step: stable (ascending token index) lists
 * of fast and slow tokens.  idx (device, 2*T int32) receives the fast list in
 * idx[0 .. n_fast) and the slow list in idx[T .. T + n_slow); counts (device,
 * 2 int32) receives {n_fast, n_slow}.  With T == 0, flags and idx may be NULL
 * and counts receives {0, 0}. */
gsi_status gsi_compact(const uint8_t* flags, int64_t T, int32_t* idx, int32_t* counts,
                       void* stream);

/* §2.2 fast and slow paths for the tokens gated by the immediately preceding
 * gsi_gate call on the same workspace, map, X and T (it reads that call's
 * counts and index lists from the workspace and its projections G):
 * Y[t] = M g_t for fast tokens, W x_t for slow tokens.  gsi_gate followed by
 * gsi_apply computes what one gsi_linear call does, in two launches that can
 * be timed separately. */
gsi_status gsi_apply(const gsi_map_desc* map, const void* X, const float* G, int64_t T,
                     float* Y, void* workspace, size_t ws_bytes, void* stream);

/* §2.1-§2.2: the gated linear map.  For each token t of X (T x d):
 * flags[t] = (rho_t >= eps); Y[t] = M g_t if fast, W x_t if slow.
 * Y: T x d_out float32 (output); flags: T bytes (output); rho: T float32
 * (output, nullable).  `workspace` holds at least
 * gsi_linear_workspace_size(map, T, GSI_PATH_AUTO) bytes, zeroed once. */
gsi_status gsi_linear(const gsi_map_desc* map, const void* X, int64_t T, float eps,
                      float* Y, uint8_t* flags, float* rho,
                      void* workspace, size_t ws_bytes, void* stream);

/* gsi_linear with an explicit choice of kernels (for comparing the decode
 * kernels with the tensor-core contractions on the same input). */
gsi_status gsi_linear_ex(const gsi_map_desc* map, const void* X, int64_t T, float eps,
                         float* Y, uint8_t* flags, float* rho,
                         void* workspace, size_t ws_bytes, gsi_path path, void* stream);

/* Workspace for gsi_stack: the maximum over its maps (the calls run in
 * stream order and reuse one workspace). */
gsi_status gsi_stack_workspace_size(const gsi_map_desc* maps, int64_t n_maps, int64_t T,
                                    size_t* bytes);

/* §2.2 "all linear maps": the gated map over a list of n_maps maps (e.g. the
 * QKV / output / MLP-up / MLP-down projections of every layer), in list
 * order, each with its own T tokens X[i] (T x maps[i].d), output Y[i]
 * (T x maps[i].d_out) and flags[i] (T bytes).  maps, X, Y, flags are HOST
 * arrays of n_maps entries; the entries are device pointers.  Outputs are not
 * chained into inputs.  Map i+1 starts reading its tokens only after map i
 * has finished, so X[i+1] may be produced by an earlier kernel of the same
 * stream. */
gsi_status gsi_stack(const gsi_map_desc* maps, int64_t n_maps, const void* const* X,
                     int64_t T, float eps, float* const* Y, uint8_t* const* flags,
                     void* workspace, size_t ws_bytes, void* stream);

/* How gsi_stack_ex runs a list of maps.
 *   AUTO / PER_MAP -- one gated-map call per map, consecutive calls chained by
 *             programmatic dependent launch (what gsi_stack does);
 *   PERSISTENT -- with one token per map, each run of consecutive maps that
 *             the single-token decode kernel takes (same element type, row
 *             width and k; at most 112) in ONE persistent launch: the maps'
 *             calls in list order, a grid barrier on the workspace between
 *             consecutive maps (map i + 1 still reads its token only after map
 *             i has finished), the next map's weights staged while the grid
 *             finishes the current one.  Outputs are bitwise those of one
 *             call per map.  Other maps, and runs the device refuses to launch
 *             co-resident, run one call each. */
typedef enum gsi_stack_mode {
  GSI_STACK_AUTO = 0,
  GSI_STACK_PER_MAP = 1,
  GSI_STACK_PERSISTENT = 2
} gsi_stack_mode;

/* gsi_stack with an explicit choice of how the list runs (same arguments,
 * results and workspace). */
gsi_status gsi_stack_ex(const gsi_map_desc* maps, int64_t n_maps, const void* const* X,
                        int64_t T, float eps, float* const* Y, uint8_t* const* flags,
                        void* workspace, size_t ws_bytes, gsi_stack_mode mode, void* stream);

/* §2.2 (Theorem 4) and §4 (static-projection control): both candidate
 * outputs of every token, for error accounting and threshold sweeps.
 * Y_fast (T x d_out float32) receives M g_t for every token (the map at
 * eps = +inf; a token with a non-finite value still takes W x_t), Y_slow
 * (T x d_out float32) receives W x_t (the map at eps = 0), rho (T float32)
 * the residual ratios, err (T float32) ||Y_fast[t] - Y_slow[t]|| and ynorm
 * (T float32) ||Y_slow[t]||.  flags (T bytes) is scratch.  All device
 * pointers; the workspace is gsi_linear's.  Enqueued on `stream`. */
gsi_status gsi_path_errors(const gsi_map_desc* map, const void* X, int64_t T, float* Y_fast, float* Y_slow,
                           uint8_t* flags, float* rho, float* err, float* ynorm, void* workspace, size_t ws_bytes,
                           void* stream);

/* §2.2: the gate at each of n_eps thresholds eps[i] (device array), from
 * gsi_path_errors' rho, err and ynorm.  n_slow[i] (int32) receives the
 * tokens with !(rho < eps[i]) (ties and NaN are slow), n_slow_calls[i] the
 * calls -- consecutive blocks of tokens_per_call tokens -- holding at least
 * one slow token (the calls that read W), and rel_err[i] (float32) the
 * gated map's relative output error against W x:
 * sqrt(sum of err^2 over fast tokens) / sqrt(sum of ynorm^2).  eps = +inf is
 * the static projection.  All device pointers; sums in double, fixed order.
 * n_eps <= 65535.  Enqueued on `stream`. */
gsi_status gsi_eps_sweep(const float* rho, const float* err, const float* ynorm, int64_t T, const float* eps,
                         int64_t n_eps, int64_t tokens_per_call, int32_t* n_slow, int32_t* n_slow_calls,
                         float* rel_err, void* stream);

/* §2.3 depth cascade and calibration.  A basis under construction is held
 * transposed and in float32: Vt is k x d, row i is basis vector i (device).
 * Readings: a layer's basis is the principal subspace of X^T X for a
 * calibration block X (T x d tokens); the next layer's basis starts from the
 * previous one and is corrected by steps V <- orthonormalise((X^T X) V),
 * the orthonormalisation being classical Gram-Schmidt in column order with
 * the DGKS test: a vector is projected a second time when its norm after a
 * projection is below 1/sqrt(2) of its norm before.  k <= GSI_MAX_K, k <= d. */

/* Orthonormalise the k rows of Vt in place (DGKS Gram-Schmidt).  n_reorth
 * (device int32, nullable) receives the number of vectors projected twice.
 * Rows that are linearly dependent on earlier ones give non-finite values. */
gsi_status gsi_basis_orthonormalize(float* Vt, int64_t k, int64_t d, int32_t* n_reorth, void* stream);

/* Bytes of `work` gsi_basis_step needs (host arithmetic; 0 for bad sizes). */
size_t gsi_basis_step_work_bytes(int64_t T, int64_t d, int64_t k);

/* One correction step on the calibration block X (T x d, element type xdt,
 * row-major, device): Vt <- DGKS((X^T (X V))^T), in place.  work: device,
 * 256-byte aligned, gsi_basis_step_work_bytes(T, d, k) bytes. */
gsi_status gsi_basis_step(const void* X, gsi_dtype xdt, int64_t T, int64_t d, int64_t k, float* Vt, void* work,
                          size_t work_bytes, int32_t* n_reorth, void* stream);

/* Subspace coherence of two orthonormal bases (Vt_a, Vt_b: k x d float32):
 * *out (device float32) = ||Va^T Vb||_F^2 / k, the mean squared cosine of the
 * principal angles (a lower bound on the mean cosine).  work: k*k floats. */
gsi_status gsi_basis_coherence(const float* Vt_a, const float* Vt_b, int64_t k, int64_t d, float* out, float* work,
                               void* stream);

/* Export a basis to a map's layout: V (d x k, row-major, dtype dt; bf16
 * rounded to nearest even) = Vt^T. */
gsi_status gsi_basis_export(const float* Vt, int64_t k, int64_t d, void* V, gsi_dtype dt, void* stream);

/* No counterpart in the paper: a library convenience.  gsi_linear for
 * callers that cannot allocate device memory (code where cudaMalloc is
 * forbidden or unavailable, such as an allocator hook, a plug-in inside a
 * host program that owns all device memory, or a loop that must never
 * allocate).  Same arguments and results as gsi_linear on the streaming
 * kernels, minus the workspace: the scratch is a built-in device array of
 * gsi_linear_noalloc_max_bytes() bytes (4 MiB) that every GPU loading the
 * library holds until the process exits.  Calls needing more scratch than
 * that (large T) return GSI_ERR_WORKSPACE.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress), so make that
 * first call before any stream capture.  Every call shares the one array:
 * calls whose executions overlap on the GPU (different streams, or host
 * threads) race and must be serialised by the caller.  Allocates nothing. */
gsi_status gsi_linear_noalloc(const gsi_map_desc* map, const void* X, int64_t T, float eps,
                              float* Y, uint8_t* flags, float* rho, void* stream);

/* Size in bytes of the built-in scratch array used by gsi_linear_noalloc. */
size_t gsi_linear_noalloc_max_bytes(void);

/* Error word of the built-in scratch (SYNCHRONISES `stream`): *code (a HOST
 * pointer) = 0 when the last gsi_linear_noalloc call on the current device
 * had no bounded device wait give up; otherwise *code is nonzero, the call's
 * outputs may be wrong and GSI_ERR_TIMEOUT is returned.  Each
 * gsi_linear_noalloc call clears the word when it starts, so query it before
 * the next call.  Allocates nothing. */
gsi_status gsi_linear_noalloc_status(uint32_t* code, void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* gsi_last_error(void);

/* Test hook: make the n-th next launch step report GSI_ERR_CUDA without
 * touching the GPU (n <= 0 disarms).  Host-side fault injection. */
void gsi_debug_fail_after(int n);

/* Test hook for the bounded waits (n <= 0 disarms): in the next n one-token
 * calls that run the single-token decode kernel's grid projection (bases
 * wider than a 16-CTA cluster holds), cluster 0 withholds its slice of g, so
 * every rank's poll for it gives up after ~10 ms instead of ~2 s.  The call
 * then completes with wrong outputs and the workspace error word set:
 * gsi_workspace_status returns GSI_ERR_TIMEOUT, and the workspace must be
 * re-initialised before its next use.  Nothing faults or hangs. */
void gsi_debug_withhold_slice(int n);

/* Test hook (n <= 0 disarms): the next n launches that need a co-resident
 * grid (the single-token decode kernel's grid projection, the two-token
 * fused kernel's grid barrier) are refused on the host, as the driver
 * refuses a grid that cannot be co-resident.  gsi_linear and gsi_stack then
 * run those calls on the two-launch streaming kernels; gsi_linear_ex with
 * GSI_PATH_FUSED returns GSI_ERR_UNSUPPORTED. */
void gsi_debug_refuse_coresident(int n);

#ifdef __cplusplus
}
#endif

#endif /* GSI_H */
