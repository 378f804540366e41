// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <vector>

#include "../../include/kfac.h"

namespace kfac {

constexpr int kNumSMs = 152;           // GB300: 2 dies x 76 SMs
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

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
  float* X;         // L^{-1} (n x n, lower; upper zero)
  float* Y;         // level scratch (n x n/2 + tile slack)
  float* Finv;      // result
  int n;
  int layer;
};

struct LayerInfo {
  int kind, o, d_in, n, has_bias, in_dtype;
  // KRON state
  size_t A, G, Ainv, Ginv, LA, LG, XA, XG, YA, YG, m;
  // DIAG state
  size_t gs, as, ticket;
  // host-side counters
  int64_t t_factor = 0, t_diag = 0;
  bool inverted = false;
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
  // K1 tensor-core operand pack (X = x-hat^T, TF32 halves or bf16)
  size_t off_tcpack = 0, tcpack_bytes = 0;
  // K4 intermediate X = dW-hat . Ainv  (o x n, max over layers)
  size_t off_k4tmp = 0, k4tmp_floats = 0;
  // K5 row-split partials and tickets
  size_t off_k5part = 0, k5part_floats = 0;
  size_t off_k5tickets = 0;
  // inversion job table (all KRON factors, sorted by n descending)
  size_t off_invjobs = 0;
  int n_invjobs = 0;
  std::vector<kfac::InvJob> invjobs_host;
  int max_kron_n = 0;

  kfac::DevStatus* status() const { return reinterpret_cast<kfac::DevStatus*>(ws + off_status); }
  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
};

namespace kfac {

// Launch bookkeeping (diagnostics): number of kernels this library launched.
void count_launch(int n = 1);
kfac_status check_launch();

// K1
kfac_status launch_update_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                  const void* g, int64_t ldg, int64_t rows, double scale,
                                  float decay, cudaStream_t s);
// K5 / K6
kfac_status launch_diag_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                const void* g, int64_t ldg, int64_t rows, double scale,
                                float* g_new, float* a_new, cudaStream_t s);
kfac_status launch_diag_step(kfac_ctx* h, int layer, float decay, const float* g_new,
                             const float* a_new, const float* gw, const float* gb, float* pw,
                             float* pb, float* ow, float* ob, cudaStream_t s);
// K2 / K3
kfac_status launch_invert(kfac_ctx* h, int layer, cudaStream_t s);
// K4
kfac_status launch_precondition(kfac_ctx* h, int layer, const float* gw, int64_t ldgw,
                                const float* gb, float* ow, float* ob, float* pw, float* pb,
                                cudaStream_t s);

// K1 on the tensor cores (tcgen05 + TMA)
kfac_status launch_syrk_tc(kfac_ctx* h, int layer, const void* x, int64_t ld, int64_t rows, int d,
                           int n, int has_bias, bool bf16, float alpha, float beta, float* F,
                           cudaStream_t st);
size_t tc_pack_bytes(int n, int64_t max_rows, bool bf16);
size_t tc_part_floats(int n, int64_t max_rows, bool bf16);

// scratch sizing helpers (used by the workspace planner)
size_t k1_scratch_floats(int n, int64_t max_rows, size_t* tickets);
size_t k5_scratch_floats(int n_plus_o, int64_t max_rows);
size_t inv_y_floats(int n);

}  // namespace kfac
