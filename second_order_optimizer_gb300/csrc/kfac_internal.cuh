// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <vector>

#include "../../include/kfac.h"

namespace kfac {

// Multiprocessor count of the current device (queried once per device).  Grids,
// split counts and the workspace plan are sized from it.
int num_sms();
// Bound on the SM count for the one statically sized scratch array
// (kfac_diag_factors_static).
constexpr int kMaxSMs = 256;
constexpr int kTcInverseMinN = 512;    // inverse assembly X^T X on the tensor cores from this n
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
// output extent of a 2-D convolution along one axis (may be < 1 for bad geometry)
inline int conv_out(int in, int k, int stride, int pad, int dil) {
  const int64_t span = (int64_t)in + 2 * (int64_t)pad - (int64_t)dil * (k - 1) - 1;
  return span < 0 ? 0 : (int)(span / stride + 1);
}

// Programmatic dependent launch.  Every library kernel is launched with the
// programmatic-serialisation attribute and starts with pdl_wait() (the grids
// before it in the stream have completed and their writes are visible; a no-op
// for an ordinary launch) and pdl_trigger() (the next grid may be scheduled
// now: its blocks do their own setup, then wait).  Each kernel waits before any
// early return, so "completed" stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Device status word: first error wins.
struct DevStatus {
  int code;    // kfac_status
  int layer;
  int info;
  int pad;
};

__device__ __forceinline__ void report_error(DevStatus* st, int code, int layer, int info) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->layer = layer;
    st->info = info;
  }
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

// One factor matrix handled by the batched inversion kernels.
struct InvJob {
  const float* F;   // running factor (n x n, symmetric)
  float* L;         // Cholesky factor, in place (n x n, lower; upper zeroed)
  float* X;         // L^{-1} (n x n, lower; the strict upper triangle stays zero
                    //   from kfac_create: no kernel writes it)
  float* Y;         // level scratch (n x n/2 + tile slack)
  float* Finv;      // result (n x n, pitch n)
  float* Finv_hi;   // result as a K4 operand, pitch np: TF32 hi and the bf16
  float* Finv_lo;   //   correction pairs of tc::corr_pair (B form)
  // inverse-free update (handles created with ikfac): K and K^T as TF32 halves,
  // and two scratch operands, all n x np; null otherwise
  float *K_hi, *K_lo, *Kt_hi, *Kt_lo, *S1_hi, *S1_lo, *S2_hi, *S2_lo;
  int n, np;
  int layer;
};

struct LayerInfo {
  int kind, o, d_in, n, has_bias, in_dtype;
  // KRON state
  size_t A, G, Ainv, Ginv, LA, LG, XA, XG, YA, YG, m;
  size_t Ainv_hi, Ainv_lo, Ginv_hi, Ginv_lo;   // pitch n_p / o_p (multiples of 4)
  size_t ik[2][8];   // ikfac: K hi/lo, K^T hi/lo, S1 hi/lo, S2 hi/lo of A (0) and G (1)
  // DIAG state
  size_t gs, as, ticket;
  // host-side counters: updates of each factor, and whether each has an inverse
  int64_t t_a = 0, t_g = 0, t_diag = 0;
  bool inv_a = false, inv_g = false;
  int tied_to = -1;   // KRON: the layer whose A (and A inverse) this layer uses, or -1
};

}  // namespace kfac

struct kfac_ctx {
  int device = 0;
  kfac_hparams hp;
  int64_t max_rows = 0;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  std::vector<kfac::LayerInfo> layers;
  size_t off_status = 0;
  // K1 split-K scratch
  size_t off_part = 0, part_floats = 0;
  size_t off_tickets = 0, n_tickets = 0;
  // the same again for the preconditioning products (SPLIT / PRECOND epilogues),
  // so factor updates and preconditioning may run concurrently on two streams
  size_t off_part_k4 = 0, off_tickets_k4 = 0;
  // K1 tensor-core operand pack (X = x-hat^T, TF32 halves or bf16)
  size_t off_tcpack = 0, tcpack_bytes = 0;
  size_t off_ones = 0;    // bf16 [ones_rows x 64]: column 0 ones, the rest zeros
  int64_t ones_rows = 0;  // 0: no such matrix (no bf16 layer with a bias)
  // K4 scratch: dW-hat halves [o x n_p] x2, then X^T halves [n x o_p] x2
  size_t off_k4tmp = 0, k4tmp_floats = 0;
  // K5 row-split partials and tickets
  size_t off_k5part = 0, k5part_floats = 0;
  size_t off_k5tickets = 0, k5tickets_ints = 0;
  // inversion job tables, three sections: [0] A then G of each KRON layer,
  // [1] the A of each, [2] the G of each (layers in order; a layer whose A is
  // tied to another's has no A job).  n_invjobs = capacity (4 per KRON layer).
  size_t off_invjobs = 0;
  int n_invjobs = 0;
  int tab_start[3] = {0, 0, 0}, tab_count[3] = {0, 0, 0};
  std::vector<kfac::InvJob> invjobs_host;
  int max_kron_n = 0;
  // inversion lookahead: the bulk of each trailing update runs on a second
  // stream, ordered against the caller's stream by two events
  cudaStream_t side_stream = nullptr;
  cudaEvent_t ev_panel = nullptr, ev_rest = nullptr;

  kfac::DevStatus* status() const { return reinterpret_cast<kfac::DevStatus*>(ws + off_status); }
  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
};

namespace kfac {

// Launch bookkeeping (diagnostics): number of kernels this library launched.
void count_launch(int n = 1);
kfac_status check_launch();

// K1
// a or g null: that factor is left as it is
kfac_status launch_update_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                  const void* g, int64_t ldg, int64_t rows, double scale,
                                  float decay_a, float decay_g, cudaStream_t s);
// K5 / K6
kfac_status launch_diag_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                const void* g, int64_t ldg, int64_t rows, double scale,
                                float* g_new, float* a_new, cudaStream_t s);
kfac_status launch_diag_factors_conv(kfac_ctx* h, int layer, const void* x, const void* gy,
                                     const kfac_conv2d_geom& geom, double scale, float* g_new,
                                     float* a_new, cudaStream_t s);
kfac_status launch_diag_step(kfac_ctx* h, int layer, float decay, const float* g_new,
                             const float* a_new, const float* gw, const float* gb, float* pw,
                             float* pb, float* ow, float* ob, cudaStream_t s);
kfac_status launch_diag_factors_batched(kfac_ctx* h, int count, const int* layers,
                                        const void* const* a, const int64_t* lda,
                                        const void* const* g, const int64_t* ldg,
                                        const int64_t* rows, double scale,
                                        float* const* g_new, float* const* a_new, cudaStream_t s);
kfac_status launch_diag_step_batched(kfac_ctx* h, int count, const int* layers,
                                     const float* decay, const float* const* g_new,
                                     const float* const* a_new, const float* const* gw,
                                     const float* const* gb, float* const* pw,
                                     float* const* pb, float* const* ow, float* const* ob,
                                     cudaStream_t s);
// geoms == nullptr: a[i], g[i] row-major with lda[i], ldg[i] (null: that factor
// is left as it is).  Otherwise a[i] is
// the NCHW input and g[i] the NCHW output gradient of the convolution geoms[i]
// (lda, ldg unused; rows[i] = batch * out_h * out_w).
kfac_status launch_update_factors_batched(kfac_ctx* h, int count, const int* layers,
                                          const void* const* a, const int64_t* lda,
                                          const void* const* g, const int64_t* ldg,
                                          const int64_t* rows, double scale,
                                          const float* decay_a, const float* decay_g,
                                          cudaStream_t s,
                                          const kfac_conv2d_geom* geoms = nullptr);
// K2 / K3: which = KFAC_FACTOR_A | KFAC_FACTOR_G; layer -1 = every KRON layer
kfac_status launch_invert(kfac_ctx* h, int layer, int which, cudaStream_t s);
// inverse-free refresh of the factors of `layer` (-1: all)
kfac_status launch_ikfac_update(kfac_ctx* h, int layer, float beta, cudaStream_t s);
// (re)write the inversion job tables on the host and the device (synchronous)
kfac_status write_inv_tables(kfac_ctx* h);
// K4
kfac_status launch_precondition(kfac_ctx* h, int layer, const float* gw, int64_t ldgw,
                                const float* gb, float* ow, float* ob, float* pw, float* pb,
                                cudaStream_t s);
kfac_status launch_precondition_batched(kfac_ctx* h, int count, const int* layers,
                                        const float* const* gw, const int64_t* ldgw,
                                        const float* const* gb, float* const* ow,
                                        float* const* ob, float* const* pw, float* const* pb,
                                        cudaStream_t s);

// Tensor-core GEMM engine (tcgen05 + TMA): C[M x N] = A[M x K] . B[N x K]^T
enum { TC_EPI_SYRK = 0, TC_EPI_SPLIT = 1, TC_EPI_PRECOND = 2 };
struct TcOperand {       // K-major operand: rows x K, row pitch in elements (16-byte multiple)
  const void* hi;        // fp32 TF32-high half, or bf16 values
  const void* lo;        // fp32 TF32-low half (unused for bf16), or with corr the
  int64_t rows, pitch;   //   bf16 correction pairs of tc::corr_pair (A or B form
  int corr;              //   by the operand's role); both operands of a product agree
};
struct TcEpilogue {
  float alpha, beta;     // SYRK: F <- beta F + alpha C (upper + mirror)
  float* C;
  int64_t ldc;
  float* out_hi;         // SPLIT: C^T stored as TF32 halves, out[c * ldo + r]
  float* out_lo;         //   (null: alpha C^T + beta out stored as fp32 in out_hi)
  int out_corr;          //   1: out_lo receives C^T's bf16 correction pairs (A form)
  int out_bf16;          //   1: alpha C^T stored as bf16 in out_hi (a bf16 array)
  int64_t ldo;
  int d_in;              // PRECOND: C = P^T (n x o): C[j][i] = P[i][j]; j >= d_in is the bias
  float eta, mu, lambda;
  float *ow, *ob, *pw, *pb, *mw, *mb;
};
kfac_status launch_gemm_tc(kfac_ctx* h, int layer, bool bf16, int epi, const TcOperand& A,
                           const TcOperand& B, bool same_ab, bool upper, int64_t M, int64_t N,
                           int64_t K, const TcEpilogue& e, cudaStream_t st, int kmode = 0);
// One product of a grouped launch.
struct TcProblem {
  TcOperand A, B;
  bool same_ab, upper;
  int64_t M, N, K;
  TcEpilogue e;
  int layer;
  // reduction range per output tile, for products with a triangular operand:
  // 0 all of K; 1 k >= the tile's first column; 2 k < the tile's last column + 1
  int kmode;
  // 3xTF32 products on CTA pairs or wide persistent tiles: k elements per TMEM
  // drain (0: the default, 128; a multiple of 32); every problem of a call the same
  int drain_k;
  // launch_syrk_direct only: A.hi is the caller's bf16 [K x A.rows] array (row
  // pitch A.pitch elements, features contiguous) read as an MN-major operand;
  // feature bias_col (a multiple of 64, or -1) reads as ones
  int bias_col;
};
// bf16 SYRKs straight from the callers' [rows x d] arrays on CTA pairs, without a
// pack: every problem has A.lo == null, same_ab, upper, M = N = n.
kfac_status launch_syrk_direct(kfac_ctx* h, const TcProblem* probs, int count, cudaStream_t st);
// Whether x can feed launch_syrk_direct: bf16, 16-byte aligned rows, a bias
// column starting its own 64-feature chunk, rows within the ones matrix.
bool syrk_direct_layout_ok(const kfac_ctx* h, const void* x, int64_t ld, int64_t rows, int d,
                           int has_bias);
// CTA-pair tiles (256 x 256) of an n x n SYRK's upper triangle.
int64_t syrk_pair_tiles(int n);
kfac_status launch_gemm_tc_grouped(kfac_ctx* h, bool bf16, int epi, const TcProblem* probs,
                                   int count, cudaStream_t st);
kfac_status launch_syrk_tc(kfac_ctx* h, int layer, const void* x, int64_t ld, int64_t rows, int d,
                           int n, int has_bias, bool bf16, float alpha, float beta, float* F,
                           cudaStream_t st);
int64_t tc_pitch(int64_t cols, bool bf16);
// one kernel whose bounded wait runs out (failure-detection self-test)
kfac_status launch_wait_selftest(kfac_ctx* h, int64_t wait_cycles, cudaStream_t st);
// Source of a gathered pack: the input patches of a 2-D convolution over an
// NCHW tensor [B, C, H, W] (output Ho x Wo), or, with a 1x1 unit-stride
// geometry, the rows of an NCHW output gradient.
struct ConvSrc {
  int B, C, H, W, kh, kw, sh, sw, ph, pw, dh, dw, Ho, Wo;
};
// x-hat -> X = x-hat^T (K-major; TF32 halves for fp32, bf16 copy), several at once.
// conv = 0: x-hat is row-major [M x d] with leading dimension ld (+ ones column);
// conv = 1: x-hat's rows are gathered from the NCHW tensor x described by cs.
struct PackJob {
  const void* x;
  int64_t ld, M;
  int d, n;
  int64_t Kp;
  void* hi;
  void* lo;
  int conv;
  ConvSrc cs;
};
constexpr int kMaxPackJobs = 32;
kfac_status launch_pack_grouped(const PackJob* jobs, int count, bool bf16, cudaStream_t st);
// Several F <- beta F + alpha x-hat^T x-hat products (fp32 inputs, 3xTF32): the
// packs of a group run as one launch and the products as grouped launches; a
// group is as many as the pack scratch holds.
struct SyrkSpec {
  const float* x;
  int64_t ld, rows;
  int d, n, layer;
  float alpha, beta;
  float* F;
  int kmode;   // TcProblem::kmode (1: x lower triangular, n x n)
};
kfac_status launch_syrk_tc_batched(kfac_ctx* h, const SyrkSpec* specs, int count, cudaStream_t st);
size_t inv_y_floats(int n);
// scratch of the batched entry points (a group of layers is packed together)
constexpr size_t kBatchScratchBudget = size_t(1) << 30;
// the batched preconditioning's gradient and X^T operands: room for every layer
// of a large set in one group (the transformer set's 24 layers take 3.2 GB), so
// that one pack and one round of product launches serve them all (transformer
// preconditioning 10.2 -> 9.9 ms with the phases in order on one stream)
constexpr size_t kPrecondScratchBudget = size_t(4) << 30;
size_t tc_pack_bytes(int n, int64_t max_rows, bool bf16);
size_t tc_part_floats();

// scratch sizing helpers (used by the workspace planner)
size_t k1_scratch_floats(int n, int64_t max_rows, size_t* tickets);
size_t k5_scratch_floats(int n_plus_o, int64_t max_rows);

}  // namespace kfac
