/*
 * kfac.h -- C ABI of the GB300 (sm_103a) Kronecker-factored optimizer step.
 *
 * The library computes, per layer, the K-FAC step described in Osawa et al.,
 * "Large-Scale Distributed Second-Order Optimization Using Kronecker-Factored
 * Approximate Curvature for Deep Convolutional Neural Networks" (§3.2: the
 * layer Fisher is approximated by the Kronecker product of a factor A built
 * from the layer's input activations and a factor G built from its output
 * gradients, and inverted through the inverses of the two factors), and the
 * fused diagonal-Fisher step of the CAFIN briefing ("CAFIN: CUDA-accelerated
 * Adaptive Fisher Information Matrix Network Optimization via GPU-Native
 * Kernel Fusion", Kernel Fusion Strategy: load gradient and parameter, update
 * the EMA of the diagonal Fisher blocks, precondition, add momentum and weight
 * decay, write the parameter in place).
 *
 * Notation per layer: d_in input width, n = d_in + has_bias (A is n x n),
 * o = d_out (G is o x o), M rows (batch; B*H_out*W_out for an unfolded
 * convolution; tokens), s = factor scale (default 1/M), xi EMA decay, gamma
 * damping, eta learning rate, mu momentum, lambda weight decay.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major.  "ld" arguments are leading dimensions in
 *     elements (>= the row length).
 *   - Every device pointer is owned by the caller.  The library allocates no
 *     device memory: all state (factors, inverses, momentum, diagonal vectors,
 *     status word) and all scratch live in the caller's workspace, whose size
 *     kfac_workspace_size() returns.  Device pointers must be aligned to their
 *     element size; 16-byte alignment enables the vectorised paths.
 *   - Work is enqueued on the given stream and the call returns without
 *     synchronising.  Only kfac_get_status() synchronises.
 *   - Argument and state errors are returned synchronously and enqueue nothing.
 *     Errors found on the device (a non positive-definite pivot, a pipeline
 *     wait that timed out) are recorded in a device status word and reported by
 *     kfac_get_status().  NaN inputs propagate; they are not checked.
 *   - A handle is not thread-safe: its calls are issued from one thread.
 *     On the device, calls on one handle must be ordered (same stream, or
 *     streams the caller orders), with one exception: the factor update
 *     (kfac_update_factors*), the preconditioning (kfac_precondition*) and
 *     the diagonal path (kfac_diag_factors*, kfac_diag_step*) use disjoint
 *     scratch and may overlap each other on different streams, as long as
 *     each touches different state (a layer's factors are read only by
 *     kfac_invert; preconditioning reads the inverses).  kfac_invert and
 *     kfac_ikfac_update must not overlap any other call on the handle: they
 *     read the factors, write the inverses, and share the factor update's
 *     and the preconditioning's scratch.
 */
#ifndef KFAC_H
#define KFAC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KFAC_OK = 0,
  KFAC_ERR_INVALID_ARG = 1,  /* bad pointer, size, layer index or hparam          */
  KFAC_ERR_WORKSPACE = 2,    /* workspace too small or misaligned                  */
  KFAC_ERR_STATE = 3,        /* e.g. precondition before the first invert          */
  KFAC_ERR_NOT_PD = 4,       /* device: damped factor not positive definite        */
  KFAC_ERR_TIMEOUT = 5,      /* device: a bounded pipeline wait gave up            */
  KFAC_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed               */
  KFAC_ERR_UNSUPPORTED = 7   /* valid request the library does not implement       */
} kfac_status;

typedef enum { KFAC_KRON = 0, KFAC_DIAG = 1 } kfac_kind;
typedef enum { KFAC_F32 = 0, KFAC_BF16 = 1 } kfac_dtype;
/* Arithmetic of the preconditioning GEMMs.  3XTF32 (fp32 accuracy): each fp32
 * operand v = h + r with h its TF32 rounding; a TF32 tensor-core product of the
 * h's plus one bf16 product that adds both cross terms h r' + r h' (from bf16
 * roundings of h and r), fp32 accumulation: the products within ~1e-6 of fp32
 * (the name is kept from the three-product form it replaces).  BF16: the inverses (rounded at each refresh), the gradient and
 * the intermediate X = dW-hat A^{-1} rounded to bf16, one bf16 tensor-core
 * product each with fp32 accumulation; factors, EMA, inverses and the
 * momentum / parameter update stay fp32 (P within ~1e-2 of fp32).  Fixed at
 * kfac_create (kfac_set_hparams rejects a change). */
typedef enum { KFAC_MATH_3XTF32 = 0, KFAC_MATH_BF16 = 1 } kfac_math;
/* Start of the running averages: ZERO gives F_1 = (1-xi) F_new; FIRST gives F_1 = F_new. */
typedef enum { KFAC_EMA_INIT_ZERO = 0, KFAC_EMA_INIT_FIRST = 1 } kfac_ema_init;

typedef struct {
  int kind;      /* kfac_kind                                                     */
  int d_out;     /* o >= 1                                                        */
  int d_in;      /* >= 1                                                          */
  int has_bias;  /* 0/1: bias is the last column of W-hat = [W | b]; a gets a ones column */
  int in_dtype;  /* kfac_dtype of the activations a and output gradients g (KRON)  */
} kfac_layer_desc;

/* Inverse-free refresh (kfac_ikfac_update): off, products in 3xTF32, or
 * products on bf16 tensor cores (fp32 accumulate and fp32 master K). */
typedef enum { KFAC_IKFAC_OFF = 0, KFAC_IKFAC_TF32 = 1, KFAC_IKFAC_BF16 = 2 } kfac_ikfac_mode;

typedef struct {
  double ema_decay;     /* xi in [0,1): F <- xi F + (1-xi) F_new                     */
  double damping;       /* gamma > 0: KRON inverts F + sqrt(gamma) I; DIAG divides by g a + gamma */
  double lr;            /* eta                                                       */
  double momentum;      /* mu                                                        */
  double weight_decay;  /* lambda: u = P + lambda W ; m <- mu m + u ; W <- W - eta m */
  int ema_init;         /* kfac_ema_init                                             */
  int math;             /* kfac_math                                                 */
  int ikfac;            /* kfac_ikfac_mode: keep inverse factors K for kfac_ikfac_update
                           (fixed at kfac_create; 32 n^2 extra workspace bytes per n x n
                           factor either way) */
} kfac_hparams;

typedef struct kfac_ctx* kfac_handle;

/* Which piece of per-layer state kfac_state_info() locates (all fp32, row-major). */
typedef enum {
  KFAC_STATE_A = 0,      /* KRON: running A, n x n, full symmetric                 */
  KFAC_STATE_G = 1,      /* KRON: running G, o x o                                 */
  KFAC_STATE_AINV = 2,   /* KRON: (A + sqrt(gamma) I)^{-1} of the latest refresh    */
  KFAC_STATE_GINV = 3,   /* KRON: (G + sqrt(gamma) I)^{-1}                          */
  KFAC_STATE_MOMENTUM = 4,  /* both: m, weight part [o x d_in] then bias part [o]  */
  KFAC_STATE_GDIAG = 5,  /* DIAG: running g diagonal, o                             */
  KFAC_STATE_ADIAG = 6   /* DIAG: running a diagonal, n                             */
} kfac_state_which;

/* Factors of a KRON layer, for kfac_invert_factors (bit mask). */
typedef enum { KFAC_FACTOR_A = 1, KFAC_FACTOR_G = 2 } kfac_factor;

/* Bytes of device workspace needed for these layers (256-byte multiple).
 * max_rows: the largest M any kfac_update_factors / kfac_diag_factors call
 * will pass for any layer (sizes the row-block scratch). */
kfac_status kfac_workspace_size(const kfac_layer_desc* layers, int n_layers,
                                const kfac_hparams* hp, int64_t max_rows, size_t* bytes);

/* Create a handle over a caller-owned workspace (>= kfac_workspace_size bytes,
 * 256-byte aligned).  Zero-fills all state (synchronously, on the legacy
 * default stream) and records the layer table.  The device that is current at
 * this call is the device of every later call. */
kfac_status kfac_create(const kfac_layer_desc* layers, int n_layers, const kfac_hparams* hp,
                        int64_t max_rows, void* d_workspace, size_t bytes, kfac_handle* out);

/* Replace the hyper-parameters (schedules such as warm-up damping, or a
 * BatchNorm damping rho_BN * gamma set around the diagonal step of those
 * layers).  Each value applies from the next call that uses it: the decay at
 * the next factor update or diagonal step, the damping at the next refresh
 * (kfac_invert*, kfac_ikfac_update) of KRON layers and the next kfac_diag_step
 * of DIAG layers, lr, momentum and weight decay at the next update.  ikfac is
 * fixed at kfac_create (a different value: KFAC_ERR_INVALID_ARG). */
kfac_status kfac_set_hparams(kfac_handle h, const kfac_hparams* hp);

/* K1: fold new factors into the running A and G of a KRON layer.
 *   A <- xi A + (1-xi) s [a 1]^T [a 1]     (ones column only if has_bias)
 *   G <- xi G + (1-xi) s g^T g
 * a: [rows x d_in] with leading dimension lda; g: [rows x d_out], ldg; both of
 * the layer's in_dtype.  scale <= 0 means s = 1/rows.  1 <= rows <= max_rows.
 * a may be NULL: A is left as it is (a stale factor, Osawa et al. §5.4, or a
 * layer whose A is tied to another's, which requires it); g may be NULL
 * likewise; not both.  With the EMA_INIT_FIRST option each factor's first
 * update replaces it.
 * Osawa et al. §3.2 (factors), §3.4 (symmetry: only the upper triangle is
 * computed; the lower is its mirror); CAFIN Introduction (EMA of the factors).
 * bf16 inputs with lda (ldg) a multiple of 8, 16-byte aligned, and (for A with a
 * bias) d_in a multiple of 64 are read in place by the tensor cores when the
 * factor fills a wave of CTA pairs (the others are first packed into the
 * workspace); the ones column then comes from a [max_rows x 64] bf16 matrix the
 * workspace holds for handles with such layers. */
kfac_status kfac_update_factors(kfac_handle h, int layer, const void* a, int64_t lda,
                                const void* g, int64_t ldg, int64_t rows, double scale,
                                cudaStream_t stream);

/* K1 for several KRON layers in one pass: the same result as calling
 * kfac_update_factors(layers[i], a[i], lda[i], g[i], ldg[i], rows[i], scale)
 * for each i, but the inputs are packed in one launch and all the factor
 * products run as one grouped tensor-core launch, so small layers fill the GPU
 * together; bf16 inputs that kfac_update_factors would read in place are read in
 * place when together they fill a wave of CTA pairs, in one further launch.
 * Host arrays of length count; each layer at most once; all layers
 * of one in_dtype.  Layers beyond what the workspace's batch scratch holds are
 * processed in further groups. */
kfac_status kfac_update_factors_batched(kfac_handle h, int count, const int* layers,
                                        const void* const* a, const int64_t* lda,
                                        const void* const* g, const int64_t* ldg,
                                        const int64_t* rows, double scale, cudaStream_t stream);

/* Geometry of a 2-D convolution (cross-correlation) over an NCHW input
 * [batch, in_channels, in_h, in_w].  The output is [batch, d_out, out_h,
 * out_w] with out = (in + 2 pad - dilation (kernel - 1) - 1) / stride + 1. */
typedef struct {
  int batch, in_channels, in_h, in_w;
  int kernel_h, kernel_w;
  int stride_h, stride_w;
  int pad_h, pad_w;
  int dilation_h, dilation_w;
} kfac_conv2d_geom;

/* K1 for a 2-D convolution layer straight from its NCHW tensors, without an
 * unfolded input:
 *   A <- xi A + (1-xi) s [P 1]^T [P 1],   G <- xi G + (1-xi) s R^T R,
 * where P [M x in_channels*kernel_h*kernel_w] holds the zero-padded input
 * patches, one row per (image b, output position oh, ow) in that order, columns
 * in the order (channel c, kernel row i, kernel column j) of a weight
 * [d_out, C, kh, kw] flattened, entry x[b, c, oh*stride_h - pad_h + i*dilation_h,
 * ow*stride_w - pad_w + j*dilation_w] (0 outside the image); R [M x d_out] holds
 * the output gradient at the same positions; M = batch*out_h*out_w.
 * x: [batch, in_channels, in_h, in_w] contiguous; gy: [batch, d_out, out_h,
 * out_w] contiguous; both of the layer's in_dtype.  scale <= 0 means s = 1/M.
 * x (gy) may be NULL to leave A (G) as it is, as in kfac_update_factors.
 * Requires d_in == in_channels*kernel_h*kernel_w, every size >= 1, pad >= 0,
 * 1 <= M <= max_rows and each tensor below 2^31 elements; otherwise
 * KFAC_ERR_INVALID_ARG before any launch.  The result equals
 * kfac_update_factors on the unfolded P and R up to the order of sums.
 * Osawa et al. §3.2 (the factors of a layer from its input activations and
 * output gradients) and §5.1 (convolutional networks: one factor row per
 * output position, M = B H_out W_out). */
kfac_status kfac_update_factors_conv2d(kfac_handle h, int layer, const void* x, const void* gy,
                                       const kfac_conv2d_geom* geom, double scale,
                                       cudaStream_t stream);

/* kfac_update_factors_conv2d for several KRON layers in one pass (one gather
 * launch for all their inputs and one grouped product launch), as
 * kfac_update_factors_batched does for row-major inputs.  Host arrays of
 * length count; each layer at most once; all layers of one in_dtype. */
kfac_status kfac_update_factors_conv2d_batched(kfac_handle h, int count, const int* layers,
                                               const void* const* x, const void* const* gy,
                                               const kfac_conv2d_geom* geoms, double scale,
                                               cudaStream_t stream);

/* K5: new diagonal factors of a layer from its a and g (any kind):
 *   g_new[i] = s sum_r g[r,i]^2 (o entries); a_new[j] = s sum_r a[r,j]^2, and
 *   a_new[d_in] = s*rows when has_bias (n entries).  Written to caller buffers.
 * CAFIN Introduction (AdaFisher's diagonal Kronecker factors). */
kfac_status kfac_diag_factors(kfac_handle h, int layer, const void* a, int64_t lda,
                              const void* g, int64_t ldg, int64_t rows, double scale,
                              float* g_new, float* a_new, cudaStream_t stream);

/* K5 for a 2-D convolution layer (any kind) from its NCHW tensors, without an
 * unfolded input: g_new[i] = s sum over (image, position) of gy[b,i,oh,ow]^2
 * (d_out entries); a_new[(c kh + i) kw + j] = s sum of the squares of the input
 * patch column (c, i, j) as in kfac_update_factors_conv2d, and a_new[d_in] =
 * s M when has_bias (n entries); s = scale, or 1/M for scale <= 0, with
 * M = batch out_h out_w.  x, gy, geom and their checks as in
 * kfac_update_factors_conv2d (both tensors required); in_h * in_w at most
 * 51200 (one channel's squares are summed in shared memory; else
 * KFAC_ERR_UNSUPPORTED).  CAFIN Introduction (the diagonal factors of
 * every layer, convolutions included); Osawa et al. §5.1. */
kfac_status kfac_diag_factors_conv2d(kfac_handle h, int layer, const void* x, const void* gy,
                                     const kfac_conv2d_geom* geom, double scale,
                                     float* g_new, float* a_new, cudaStream_t stream);

/* K5 for several layers in one launch: the same result as calling
 * kfac_diag_factors(layers[i], a[i], lda[i], g[i], ldg[i], rows[i], scale,
 * g_new[i], a_new[i]) for each i, up to the order of the floating-point sums
 * over rows (each column is still summed with compensation, then the row
 * splits in fixed order).  Host arrays of length count; each layer at most
 * once; all layers of one in_dtype.  Groups beyond the workspace's K5 scratch
 * or 64 layers are processed in further launches. */
kfac_status kfac_diag_factors_batched(kfac_handle h, int count, const int* layers,
                                      const void* const* a, const int64_t* lda,
                                      const void* const* g, const int64_t* ldg,
                                      const int64_t* rows, double scale, float* const* g_new,
                                      float* const* a_new, cudaStream_t stream);

/* K2+K3: damped inverses (F + sqrt(gamma) I)^{-1} for F in {A, G} of one KRON
 * layer, or of every KRON layer when layer == -1 (one batched pass), by
 * blocked Cholesky and a blocked triangular inverse.  A non positive-definite
 * pivot sets KFAC_ERR_NOT_PD in the status word (layer, 0-based column).
 * Osawa et al. §3.2 (inverse through the factor inverses), §5.4 (refresh
 * every few steps, so this call is made every k-th step by the caller). */
kfac_status kfac_invert(kfac_handle h, int layer, cudaStream_t stream);

/* K2+K3 for a chosen factor: which = KFAC_FACTOR_A, KFAC_FACTOR_G or both
 * (bit or).  The same as kfac_invert restricted to those factors, so A and G
 * may be refreshed on their own cadences (Osawa et al. §5.4: after a warm-up
 * the refreshes are made rarer, and A, which fluctuates less than G, may be
 * refreshed less often).  A factor not refreshed keeps the inverse of its
 * latest refresh.  A layer whose A is tied (kfac_tie_a_factor) has no A of its
 * own: KFAC_FACTOR_A is ignored for it (its source's refresh covers it).
 * which outside 1..3: KFAC_ERR_INVALID_ARG. */
kfac_status kfac_invert_factors(kfac_handle h, int layer, int which, cudaStream_t stream);

/* Inverse-free refresh ("Structured Inverse-Free Natural Gradient" page,
 * abstract: an inverse-free K-FAC update that subtracts in the matrix-logarithm
 * space instead of inverting).  For each factor F of the layer (or of every
 * KRON layer, layer == -1) the handle keeps K with K K^T standing for
 * (F + sqrt(gamma) I)^{-1}; one call takes the step
 *   K <- K (I - (beta/2) (K^T (F + sqrt(gamma) I) K - I)),
 * the first-order form of K exp(-(beta/2) E) (E vanishes at the exact inverse),
 * and sets the layer's inverse to K K^T, which kfac_precondition then uses.
 * Every product runs on the tensor cores; no factorisation.  With
 * hp->ikfac = KFAC_IKFAC_TF32 the products are 3xTF32 (fp32 accuracy).  With
 * KFAC_IKFAC_BF16 (the page: stable in low precision) they run on bf16 tensor
 * cores with fp32 accumulation: K^T is kept in fp32 and gains the step's
 * correction -(beta/2) K E in fp32, F + sqrt(gamma) I enters as a bf16 hi/lo
 * pair, and K K^T is a bf16 SYRK (inverses within ~5e-3 of the fp64 iteration
 * on the tests' factors).  K is seeded by each kfac_invert of the factor
 * (K = L^{-T}, exactly the inverse factor), so a factor needs one kfac_invert
 * before its first update.
 * Requires a handle created with hp->ikfac != 0 (else KFAC_ERR_UNSUPPORTED),
 * 0 < beta < 2 (else KFAC_ERR_INVALID_ARG), and an inverted factor (else
 * KFAC_ERR_STATE).  A tied A is stepped with its source.  Like kfac_invert,
 * it must not overlap other calls of the handle. */
kfac_status kfac_ikfac_update(kfac_handle h, int layer, double beta, cudaStream_t stream);

/* Tie layer's A factor to source's: from now on `layer` uses source's running
 * A and A inverse (kfac_state_info reports source's), has no A update or
 * inversion of its own, and its kfac_update_factors* calls must pass a NULL
 * a (any other a: KFAC_ERR_INVALID_ARG).  For layers fed the same input (the
 * query, key and value projections of an attention block), whose A factors
 * are identical: the factor is built and inverted once.  Both KRON layers of
 * the same n = d_in + has_bias, layer != source, source not itself tied, no
 * layer tied to `layer`, and no factor update or inversion made yet on either
 * (else KFAC_ERR_INVALID_ARG or KFAC_ERR_STATE).  Synchronous: rewrites the
 * handle's inversion tables on the device, so call it before any work is
 * enqueued on the handle.  Osawa et al. §3.2 (A is built from the layer's
 * input activations alone). */
kfac_status kfac_tie_a_factor(kfac_handle h, int layer, int source);

/* K4: preconditioned gradient P = Ginv . [dW | db] . Ainv of a KRON layer.
 * grad_w: [o x d_in] fp32, ld ldgw; grad_b: [o] (required iff has_bias).
 * out_w [o x d_in] (ld d_in) / out_b [o]: P, nullable when param_w is given.
 * param_w [o x d_in] (ld d_in) / param_b [o]: nullable; when given the update
 *   u = P + lambda W ; m <- mu m + u ; W <- W - eta m   is applied in place
 * (m is library state).  Returns KFAC_ERR_STATE until both of the layer's
 * inverses exist (for a tied A, its source's).  CAFIN Kernel Fusion Strategy
 * (precondition, momentum, weight
 * decay, in-place write); Osawa et al. §3.2. */
kfac_status kfac_precondition(kfac_handle h, int layer, const float* grad_w, int64_t ldgw,
                              const float* grad_b, float* out_w, float* out_b,
                              float* param_w, float* param_b, cudaStream_t stream);

/* K4 for several KRON layers in one pass: the same result as calling
 * kfac_precondition for each i with the i-th entries of the host arrays
 * (grad_b, out_w, out_b, param_w, param_b may be NULL arrays, or hold NULL
 * entries, under the same rules as the single call).  Each layer at most once.
 * The gradients are packed in one launch and each of the two products runs
 * as one grouped tensor-core launch over the layers. */
kfac_status kfac_precondition_batched(kfac_handle h, int count, const int* layers,
                                      const float* const* grad_w, const int64_t* ldgw,
                                      const float* const* grad_b, float* const* out_w,
                                      float* const* out_b, float* const* param_w,
                                      float* const* param_b, cudaStream_t stream);

/* K6: fused diagonal-Fisher step of a DIAG layer, one streaming pass:
 *   gs <- xi gs + (1-xi) g_new ; as <- xi as + (1-xi) a_new     (library state)
 *   P_ij = [dW | db]_ij / (gs_i as_j + gamma)
 *   u = P + lambda W ; m <- mu m + u ; W <- W - eta m           (W in place)
 * g_new [o], a_new [n] (e.g. from kfac_diag_factors, or supplied by the caller
 * for BatchNorm: o = channels, d_in = 1, has_bias = 1, W = scale, b = shift).
 * grad_w/param_w: [o x d_in] contiguous; grad_b/param_b: [o] iff has_bias.
 * out_w/out_b: optional copy of P (nullable).  CAFIN Kernel Fusion Strategy;
 * Osawa et al. §5.4 (BatchNorm Fisher taken as diagonal). */
kfac_status kfac_diag_step(kfac_handle h, int layer, const float* g_new, const float* a_new,
                           const float* grad_w, const float* grad_b,
                           float* param_w, float* param_b, float* out_w, float* out_b,
                           cudaStream_t stream);

/* K6 for several DIAG layers in one streaming launch: bit-for-bit the result
 * of calling kfac_diag_step for each i with the i-th entries of the host
 * arrays (grad_b, param_b, out_w, out_b may be NULL arrays or hold NULL
 * entries under the same rules as the single call).  Each layer at most once;
 * up to 64 layers per launch, more in further launches.  One ticket orders the
 * write-back of every layer's EMA vectors after all reads. */
kfac_status kfac_diag_step_batched(kfac_handle h, int count, const int* layers,
                                   const float* const* g_new, const float* const* a_new,
                                   const float* const* grad_w, const float* const* grad_b,
                                   float* const* param_w, float* const* param_b,
                                   float* const* out_w, float* const* out_b,
                                   cudaStream_t stream);

/* Failure-detection self-test: enqueue one kernel that waits, through the
 * same bounded mbarrier wait every pipeline role of the library uses, for a
 * phase that nothing completes.  The wait gives up after wait_cycles SM clocks
 * (1 <= wait_cycles <= 2^31; the library's own waits give up after 2e9, about
 * a second), records KFAC_ERR_TIMEOUT in the status word (layer -1, info 1)
 * and the kernel returns: no fault, trap or endless loop, and the context
 * stays usable.  kfac_get_status() then reports (and clears) it. */
kfac_status kfac_selftest_timeout(kfac_handle h, int64_t wait_cycles, cudaStream_t stream);

/* Synchronise the device and report the first device-side error since the
 * last call (then clear it).  bad_layer / info (nullable) receive the layer
 * and, for KFAC_ERR_NOT_PD, the 0-based column of the failing pivot. */
kfac_status kfac_get_status(kfac_handle h, int* bad_layer, int* info);

/* Byte offset (within the workspace) and size of one piece of layer state,
 * for checkpointing through the caller's own copies. */
kfac_status kfac_state_info(kfac_handle h, int layer, int which, size_t* offset, size_t* bytes);

/* Release the handle (host memory only; the workspace stays the caller's). */
kfac_status kfac_destroy(kfac_handle h);

/* Static description of a status code. */
const char* kfac_status_string(kfac_status s);

/* K5 without a handle or workspace, for callers that cannot allocate device
 * memory (no cudaMalloc, no caller-provided workspace): for instance code that
 * runs under another framework's allocator, or a plug-in whose host owns all
 * device allocations.  The paper has no counterpart to this entry point; it
 * computes exactly what kfac_diag_factors computes for a layer with these
 * dimensions (same kernel; on GPUs with at most 256 SMs the same row splits and
 * so the same results).
 * Scratch: a static device array of 1.5 MiB (partial sums) plus 4 KiB
 * (counters) that every GPU which loads the library keeps until process exit.
 * Limit: d_in + d_out <= 262144, else KFAC_ERR_WORKSPACE.  Allocates nothing:
 * no cudaMalloc/cudaFree, no allocating library call.  Each call looks up the
 * array's device address on the current device (a host-side query; the first
 * call on a device may load the library's device code there, so make it before
 * any stream capture).  Every call shares the one array and it
 * keeps the last call's contents: calls that overlap on the GPU (other
 * streams, other threads) race; order them.  Arguments as kfac_diag_factors
 * plus the layer shape: in_dtype is a kfac_dtype, scale <= 0 means 1/rows. */
kfac_status kfac_diag_factors_static(const void* a, int64_t lda, const void* g, int64_t ldg,
                                     int64_t rows, int d_in, int d_out, int has_bias,
                                     int in_dtype, double scale, float* g_new, float* a_new,
                                     cudaStream_t stream);

/* Diagnostics: number of kernels this library has launched in this process. */
unsigned long long kfac_launch_count(void);

/* Diagnostics: the CUDA runtime's description of the last launch error behind a
 * KFAC_ERR_CUDA return in this process ("no error" if there was none).  Static
 * string; not cleared by later successful calls. */
const char* kfac_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* KFAC_H */
