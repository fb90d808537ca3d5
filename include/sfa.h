/*
 * sfa.h -- C ABI of libsfa, depth-staggered Fibonacci sparse attention on
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the attention of "Depth-Staggered Fibonacci Spacing for
 * Sparse Attention: Static Schedules Beat Learned Dilation and Extrapolate
 * Where Dense Attention Fails" (arXiv 2606.28560), section 2 "Method":
 *
 *   For query i the attended keys are the dense window of distances 0..W
 *   (self included) and one "rung" per base offset f_k at the continuous
 *   distance d_k = alpha * f_k.  A rung reads key and value row i - d_k by
 *   linear interpolation between rows i - floor(d_k) (weight 1 - t) and
 *   i - floor(d_k) - 1 (weight t), t = d_k - floor(d_k).  RoPE is applied at
 *   the true positions before that gather.  The offsets are shared by all
 *   queries (a shift, not a per-position index list).  One softmax runs over
 *   the union of window and rung entries.  The per-layer scalar is
 *   alpha = 0.5 + sigmoid(theta) ("Per-layer scalar").
 *
 * Conventions fixed by this library where the paper is silent:
 *   - d_k is the fp32 product fl32(alpha) * fl32(f_k), rounded to nearest;
 *   - a rung with d_k <= W is dropped (its distance is in the window);
 *   - a rung is masked for query i when i - ceil(d_k) < 0;
 *   - RoPE pairs dimension m with m + D/2 ("rotate half"), angle
 *     pos * rope_theta^(-2m/D);
 *   - query head h reads key/value head h / (Hq / Hkv);
 *   - the softmax scale defaults to 1/sqrt(D).
 *
 * Layouts.  Q, O, dO, dQ: [B][T][Hq][D]; K, V, dK, dV: [B][T][Hkv][D]; all
 * row-major with D fastest, element type sfa_params.dtype.  lse: [B][T][Hq]
 * fp32 (natural-log log-sum-exp of the scaled scores).  All tensors are
 * device pointers aligned to 16 bytes and must not overlap one another.
 *
 * Ownership.  The caller allocates every buffer (outputs, workspace, RoPE
 * table, status word).  The library allocates no device or host memory and
 * carries no data from one call to the next; the rung table is copied into
 * the kernel arguments.  What it keeps is per device and read-only after the
 * first call there: the SM count, kernel attributes already set, resident
 * CTAs per SM of its persistent kernels, and sfa_forward_noalloc's fixed
 * scratch array (part of the library image).  Every call is asynchronous on
 * the given stream and returns before the GPU finishes.
 *
 * Errors.  Invalid arguments return SFA_ERR_INVALID_ARG and shapes outside the
 * supported set return SFA_ERR_UNSUPPORTED, both before anything is launched.
 * A failed launch returns SFA_ERR_CUDA.  A kernel that gives up a bounded wait
 * sets a bit in the optional device status word (see SFA_DEVSTAT_*) and
 * returns; sfa_read_status() turns a non-zero word into SFA_ERR_DEVICE_STATUS.
 * Outputs are undefined after any error.
 *
 * Test hook.  With SFA_TEST_FAULT=launch in the environment (read once per
 * process) every entry point that would launch work or read the status word
 * checks its arguments as usual and then returns SFA_ERR_CUDA without
 * launching, so that a caller's error handling can be exercised without
 * faulting a GPU.  Calls with nothing to launch (B * T = 0) still return
 * SFA_OK, except sfa_backward, which then still zeroes dalpha and dtheta and
 * so fails too.
 */
#ifndef SFA_H
#define SFA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SFA_API __attribute__((visibility("default")))
#else
#define SFA_API
#endif

#define SFA_MAX_RUNGS 32

typedef enum {
    SFA_OK = 0,
    SFA_ERR_INVALID_ARG = 1,
    SFA_ERR_UNSUPPORTED = 2,
    SFA_ERR_CUDA = 3,
    SFA_ERR_DEVICE_STATUS = 4
} sfa_status;

typedef enum { SFA_F32 = 0, SFA_BF16 = 1 } sfa_dtype;

/* Bits a kernel may set in the device status word. */
#define SFA_DEVSTAT_WAIT_TIMEOUT 0x1u  /* a bounded pipeline wait gave up */
#define SFA_DEVSTAT_BAD_INDEX    0x2u  /* a computed row index left [0, T) */

typedef struct {
    int B, T;          /* batch, sequence length (>= 0; 0 means nothing to do);
                          T <= 2^24 and B * T <= 2^28, else SFA_ERR_UNSUPPORTED */
    int Hq, Hkv, D;    /* heads and head dim; supported: Hq = 8, Hkv = 2, D = 64 */
    int W;             /* window: distances 0..W (W >= 0) */
    int K;             /* number of base offsets, 0 <= K <= SFA_MAX_RUNGS */
    const float *rungs;/* HOST pointer to K base offsets f_k (finite, > 0) */
    float alpha;       /* the layer's scalar (finite, > 0) */
    float rope_theta;  /* RoPE base (1e4 in the paper); <= 0: inputs already rotated */
    float scale;       /* softmax scale; 0 selects 1/sqrt(D).  Accuracy with
                          bf16 and rope_theta > 0: the rotated query and key
                          rows are rounded to bf16 before they are scored, so
                          a score s = scale q.k carries an error of up to
                          about scale |q| |k| 2^-7 (Cauchy-Schwarz bound; the
                          typical error is about 2^-8 scale |q| |k| / sqrt(D)).
                          For inputs of unit scale this rounding alone
                          moves O and LSE by about 0.007 at the default scale
                          1/8 and by about 0.02 at scale 0.3 (600 query rows
                          measured); sharper scores (a larger scale or larger
                          norms) move LSE by up to that bound.  fp32, or bf16
                          without RoPE, scores the given values exactly. */
    sfa_dtype dtype;   /* element type of Q, K, V, O, dO, dQ, dK, dV */
    int round_offsets; /* 0: d_k as computed (interpolated gather); 1: every d_k
                          rounded to the nearest integer, halves up (the static
                          schedules "with integer offsets", section 2
                          "Implementation notes"): one row per rung, and
                          dL/dalpha = 0 */
} sfa_params;

/* Library version, (major << 16) | minor. */
SFA_API int sfa_version(void);

/* Human-readable name of a status code (static string). */
SFA_API const char *sfa_strerror(sfa_status s);

/* Number of kernels this library has launched in the process so far (host
 * counter, incremented on every successful launch). */
SFA_API unsigned long long sfa_launch_count(void);

/* ---- per-layer scalar ("Per-layer scalar", section 2) ---------------- */

typedef enum {
    SFA_SCHEDULE_FIXED = 0,   /* alpha_l = 1 */
    SFA_SCHEDULE_LEARNED = 1, /* alpha_l = 0.5 + sigmoid(theta_l) */
    SFA_SCHEDULE_LINEAR = 2,  /* alpha_l = 0.5 + l / (L - 1) */
    SFA_SCHEDULE_COPRIME = 3  /* linear ramp re-assigned by l -> (S l) mod L */
} sfa_schedule;

/* alpha = 0.5 + sigmoid(theta), computed in double and rounded to float. */
SFA_API float sfa_alpha_from_theta(float theta);

/* Fills alpha_out[0..L-1] (host) with the schedule's per-layer scalars.
 * theta (host, L values) is read only by SFA_SCHEDULE_LEARNED; S is the
 * coprime stride (7 in the paper) and must satisfy gcd(S, L) = 1.
 * Values are computed in double and rounded once to float. */
SFA_API sfa_status sfa_alpha_schedule(sfa_schedule kind, int L, int S,
                                      const float *theta, float *alpha_out);

/* ---- rung preparation (host; "Attended set", section 2) -------------- */

/* The rungs the kernels will use for this layer, by increasing distance: for
 * every base offset with d_k = fl32(alpha) * fl32(f_k) > W and
 * ceil(d_k) <= T - 1 (rungs beyond that are masked for every query) it
 * reports the table index, floor(d_k), t = d_k - floor(d_k) and ceil(d_k)
 * (with p->round_offsets, d_k is first rounded to the nearest integer, halves
 * up, so that t = 0 and floor = ceil).
 * Arrays are host arrays of at least p->K entries; *n_active receives the
 * count.  This is the same routine sfa_forward and sfa_backward use. */
SFA_API sfa_status sfa_rung_plan(const sfa_params *p, int *n_active, int *index,
                                 int *n_floor, float *frac, int *n_ceil);

/* ---- RoPE table ------------------------------------------------------ */

/* Number of floats of a RoPE table for T positions and head dim D (T * D). */
SFA_API size_t sfa_rope_table_floats(int T, int D);

/* Writes the RoPE table on the device: table[pos][m] = (cos, sin) of
 * pos * rope_theta^(-2m/D) for pos < T, m < D/2, as float pairs, angles and
 * trigonometry in double.  The table serves every call with the same D and
 * rope_theta and a sequence length <= T.  table: device, 16-byte aligned,
 * sfa_rope_table_floats(T, D) floats. */
SFA_API sfa_status sfa_rope_table(float *table, int T, int D, float rope_theta,
                                  cudaStream_t stream);

/* ---- forward ----------------------------------------------------------- */

/* Bytes of device workspace sfa_forward needs (0 when it needs none).  The
 * bf16 path keeps the rotated keys there: B * T * Hkv * D * 2 bytes. */
SFA_API size_t sfa_forward_workspace_size(const sfa_params *p);

/* O = sparse attention(Q, K, V) for one layer (section 2 "Attended set").
 *   Q [B][T][Hq][D], K and V [B][T][Hkv][D] (device, dtype p->dtype);
 *   rope_table: from sfa_rope_table with >= T positions, p->D and
 *     p->rope_theta; may be NULL only when p->rope_theta <= 0;
 *   O [B][T][Hq][D] (device, dtype p->dtype), fully overwritten;
 *   lse [B][T][Hq] fp32 (device) or NULL; required by sfa_backward;
 *   workspace: device, 256-byte aligned, >= sfa_forward_workspace_size(p)
 *     bytes (may be NULL when that size is 0), clobbered;
 *   status: device word or NULL (see SFA_DEVSTAT_*).
 * bf16: RoPE on the keys (one launch, skipped when rope_theta <= 0), then the
 * tensor-core attention kernel (one launch), for W <= 30; fp32 and wider
 * windows: one fp32-arithmetic kernel.  Asynchronous on stream. */
SFA_API sfa_status sfa_forward(const sfa_params *p, const void *Q, const void *K,
                               const void *V, const float *rope_table, void *O,
                               float *lse, void *workspace, size_t workspace_bytes,
                               unsigned int *status, cudaStream_t stream);

/* ---- forward of several layers ----------------------------------------- */

/* Bytes of device workspace sfa_forward_layers needs for L layers (windows:
 * host array of L windows, or NULL for p->W in every layer). */
SFA_API size_t sfa_forward_layers_workspace_size(const sfa_params *p, int L, const int *windows);

/* The forwards of L layers of a model in one call (the paper's model has 16
 * attention layers, each with its own scalar alpha_l: section 2 "Per-layer
 * scalar", section 3 "Model and training").  Layer l computes exactly what
 * sfa_forward computes with *p, alpha = alphas[l] and W = windows[l] (p->W
 * when windows is NULL) on Q[l], K[l], V[l] into O[l] and lse[l].
 *   alphas, windows: host arrays of L values; p->alpha is not read;
 *   Q, K, V, O: host arrays of L device pointers (layouts as sfa_forward);
 *   lse: host array of L device pointers (entries may be NULL) or NULL;
 *   workspace: device, 256-byte aligned, >= sfa_forward_layers_workspace_size
 *     bytes, clobbered; status: as sfa_forward.
 * When every layer takes the bf16 tensor-core path with RoPE, the call makes
 * one RoPE launch for layer 0's keys and one attention launch per layer, and
 * each attention launch also rotates the next layer's keys (two rotated-key
 * buffers in the workspace, used in turn); otherwise it is L sfa_forward
 * calls.  Arguments of every layer are checked before anything is launched;
 * errors as sfa_forward.  Asynchronous on stream. */
SFA_API sfa_status sfa_forward_layers(const sfa_params *p, int L, const float *alphas,
                                      const int *windows, const void *const *Q,
                                      const void *const *K, const void *const *V,
                                      const float *rope_table, void *const *O, float *const *lse,
                                      void *workspace, size_t workspace_bytes,
                                      unsigned int *status, cudaStream_t stream);

/* ---- forward without a caller workspace ------------------------------- */

/* The paper has no counterpart to this entry point: it serves callers that
 * cannot allocate device memory (a plugin in a host application that owns all
 * device memory, a fixed-footprint service, a tool limited to memory reserved
 * up front).  It computes exactly what sfa_forward computes, with the same
 * arguments minus the workspace: the bf16 path's rotated keys go to a fixed
 * array inside the library, of sfa_forward_noalloc_scratch_bytes() bytes
 * (8 MiB, enough for B * T <= 32768 tokens at Hkv = 2, D = 64), which every
 * GPU that loads the library holds until the process exits.
 *   - Returns SFA_ERR_UNSUPPORTED, before any launch, when the shape needs
 *     more scratch than that; other errors as sfa_forward.
 *   - Allocates nothing.  The first call in each CUDA context (a device's
 *     primary context, or one the caller created with cuCtxCreate and made
 *     current) looks the array's device address up with cudaGetSymbolAddress
 *     in that context and caches it under the context's id (cuCtxGetId, never
 *     reused within a process), so every call uses the address valid in the
 *     context it is made from.  Make the first call in each context before
 *     any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race on it and give wrong results; order them
 *     on one stream.  Nothing in the array needs to start at zero. */
SFA_API size_t sfa_forward_noalloc_scratch_bytes(void);

SFA_API sfa_status sfa_forward_noalloc(const sfa_params *p, const void *Q, const void *K,
                                       const void *V, const float *rope_table, void *O,
                                       float *lse, unsigned int *status, cudaStream_t stream);

/* ---- fused front end: QKV projection with RoPE ---------------------- */

/* The step before the attention of a layer (section 3 "Model and training":
 * d_model 512, 8 query and 2 key/value heads of dimension 64; section 2
 * "Attended set": RoPE at the true positions before any key row is
 * gathered): [Q | K | V] = X . Wqkv^T, then Q and K rotated,
 *   Qhat[b][i][h][:] = R(i) Q[b][i][h][:],  Khat[b][i][g][:] = R(i) K[b][i][g][:],
 * R(i) the rotate-half rotation of pairs (m, m + 32) by the angle
 * i * rope_theta^(-2m/64) (the table of sfa_rope_table).  sfa_forward with
 * rope_theta = 0 then computes the same attention as sfa_forward on the
 * unrotated Q, K with rope_theta set.
 *   p: B, T, Hq = 8, Hkv = 2, D = 64, dtype SFA_BF16 and rope_theta are used
 *     (rope_theta = 0: no rotation, a plain projection); the other fields are
 *     validated as for sfa_forward but not used;
 *   d_model: a multiple of 64, 64 .. 16384;
 *   X [B][T][d_model] bf16, row-major;
 *   Wqkv [768][d_model] bf16, row-major (the weight of a linear layer): rows
 *     64h .. 64h + 63 produce query head h (h < 8), rows 512 + 64g .. key
 *     head g, rows 640 + 64g .. value head g (g < 2); row r of a block is
 *     dimension r mod 64;
 *   rope_table: >= T positions (device, from sfa_rope_table); NULL when
 *     rope_theta = 0;
 *   Qhat [B][T][8][64], Khat [B][T][2][64], V [B][T][2][64] bf16 (outputs,
 *     natural dimension order);
 *   status: device word or NULL (SFA_DEVSTAT_WAIT_TIMEOUT if a pipeline wait
 *     gave up; the outputs are then not written).
 * All device pointers 16-byte aligned.  One launch on the tensor cores
 * (tcgen05, fp32 accumulation in tensor memory); allocates nothing.
 * Asynchronous on stream. */
SFA_API sfa_status sfa_qkv_rope(const sfa_params *p, int d_model, const void *X, const void *Wqkv,
                                const float *rope_table, void *Qhat, void *Khat, void *V,
                                unsigned int *status, cudaStream_t stream);

/* ---- failure-path self-test ------------------------------------------- */

/* Exercises the failure path that the pipelined kernels share: every wait on
 * an mbarrier gives up after a fixed limit (0.25 s), sets the CTA's abort
 * flag so the other warps leave their waits, and sets
 * SFA_DEVSTAT_WAIT_TIMEOUT in the status word; the kernel then returns and
 * the context stays usable.  One CTA waits, with those same wait routines, on
 * a barrier that nothing arrives on.  Touches no data.
 *   status: device word (required, 4-byte aligned); SFA_DEVSTAT_WAIT_TIMEOUT
 *     is set in it when the call has run (after about 0.25 s).
 * One launch; asynchronous on stream. */
SFA_API sfa_status sfa_selftest_wait_timeout(unsigned int *status, cudaStream_t stream);

/* ---- decode ------------------------------------------------------------ */

/* One new query per sequence over a key/value cache: the attention of query
 * i = positions[b] of sequence b (section 2 "Attended set"), as sfa_forward
 * computes it for row (b, i), reading only cache rows 0..i.  This is the
 * inference workload of the paper's latency comparison between the
 * interpolated gather and integer offsets (section 3 "Run matrix", section
 * 4.3).
 *   p->B: sequences; p->T: cache capacity Tc (>= 1); other fields as
 *     sfa_forward (the rung plan is made for a sequence of length Tc);
 *   Q [B][Hq][D]: the new tokens' queries (unrotated when rope_theta > 0);
 *   Kc, Vc [B][Tc][Hkv][D]: the cache, row i of sequence b holding the new
 *     token's own key and value (keys unrotated when rope_theta > 0);
 *   positions: device int32 [B]; a position outside [0, Tc) reads nothing,
 *     writes zeros to that sequence's outputs and sets SFA_DEVSTAT_BAD_INDEX
 *     in *status;
 *   rope_table: >= Tc positions (as sfa_forward); O [B][Hq][D];
 *   lse [B][Hq] fp32 or NULL.
 * One launch (fp32 arithmetic for both dtypes); allocates nothing.
 * Asynchronous on stream. */
SFA_API sfa_status sfa_decode(const sfa_params *p, const void *Q, const void *Kc,
                              const void *Vc, const int *positions, const float *rope_table,
                              void *O, float *lse, unsigned int *status, cudaStream_t stream);

/* ---- backward ---------------------------------------------------------- */

/* Bytes of device workspace sfa_backward needs for these parameters. */
SFA_API size_t sfa_backward_workspace_size(const sfa_params *p);

/* Gradients of a scalar loss L given dO = dL/dO (section 2 "Implementation
 * notes": the interpolation fraction carries the gradient to alpha).
 *   Q, K, V, O, dO: as in sfa_forward (O from sfa_forward with the same
 *     arguments); lse: from that forward (required);
 *   dQ [B][T][Hq][D], dK and dV [B][T][Hkv][D]: device, dtype p->dtype,
 *     fully overwritten;
 *   dalpha: device, 1 float, receives dL/dalpha = sum_k f_k * dL/dt_k;
 *   dtheta: device, 1 float, receives dL/dalpha * (alpha - 0.5) * (1.5 - alpha),
 *     the gradient to theta when alpha = 0.5 + sigmoid(theta);
 *   workspace: device, 256-byte aligned, >= sfa_backward_workspace_size(p)
 *     bytes, contents ignored on entry and clobbered;
 *   status: device word or NULL.
 * The derivative of floor/ceil and of the drop and mask decisions is zero.
 * Asynchronous on stream.  bf16 with W <= 30: three launches (one that
 * zeroes the fp32 accumulators in the workspace and rotates K, the rotation
 * skipped when rope_theta <= 0; the tensor-core kernel; a finish launch);
 * fp32 and wider windows: three launches of the fp32-arithmetic kernels. */
SFA_API sfa_status sfa_backward(const sfa_params *p, const void *Q, const void *K,
                                const void *V, const void *O, const void *dO,
                                const float *lse, const float *rope_table, void *dQ,
                                void *dK, void *dV, float *dalpha, float *dtheta,
                                void *workspace, size_t workspace_bytes,
                                unsigned int *status, cudaStream_t stream);

/* ---- device status ----------------------------------------------------- */

/* Synchronises stream, copies the device status word to *host_word (may be
 * NULL) and returns SFA_ERR_DEVICE_STATUS if it is non-zero, SFA_OK if zero. */
SFA_API sfa_status sfa_read_status(const unsigned int *status, unsigned int *host_word,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SFA_H */
