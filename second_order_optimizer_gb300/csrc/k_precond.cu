// K4: natural-gradient direction P = Ginv . [dW | db] . Ainv, with the optional fused update
//     u = P + lambda W ;  m <- mu m + u ;  W <- W - eta m      (in place).
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", §3.2 (the inverse Fisher is
// applied through the two factor inverses, one on each side of the weight
// gradient).  "CAFIN: CUDA-accelerated Adaptive Fisher Information Matrix
// Network Optimization via GPU-Native Kernel Fusion", Kernel Fusion Strategy
// (precondition, then momentum and weight decay, then the in-place write),
// fused here into the epilogue of the second product.
//
// Both products run on the tensor cores in 3xTF32 (fp32 accuracy):
//   pack     dW-hat = [dW | db] -> TF32 halves [o x n_p]
//   X^T  =   Ainv . dW-hat^T      M = n, N = o, K = n   epilogue stores X^T as TF32 halves
//   P    =   Ginv . X             M = o, N = n, K = o   epilogue: P out and/or W, m update
// Writing X^T (not X) keeps every operand K-major.  Ainv/Ginv halves are
// produced once per refresh by the inverse pass.
#include "kfac_internal.cuh"
#include "tc_prims.cuh"

#include <algorithm>

namespace kfac {

namespace {

__global__ void __launch_bounds__(256) gradhat_pack_kernel(const float* __restrict__ gw, int64_t ld,
                                                           const float* __restrict__ gb, int o,
                                                           int d_in, int n, int64_t np,
                                                           float* hi, float* lo) {
  const int64_t total = (int64_t)o * n;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = e / n, j = e % n;
    const float v = j < d_in ? gw[i * ld + j] : gb[i];
    const float h = tc::to_tf32(v);
    hi[i * np + j] = h;
    lo[i * np + j] = tc::to_tf32(v - h);
  }
}

}  // namespace

kfac_status launch_precondition(kfac_ctx* h, int layer, const float* gw, int64_t ldgw,
                                const float* gb, float* ow, float* ob, float* pw, float* pb,
                                cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  const int64_t np = tc_pitch(L.n, false), op = tc_pitch(L.o, false);
  if ((size_t)(2 * L.o * np + 2 * L.n * op) > h->k4tmp_floats) return KFAC_ERR_WORKSPACE;
  float* g_hi = h->at<float>(h->off_k4tmp);
  float* g_lo = g_hi + (size_t)L.o * np;
  float* x_hi = g_lo + (size_t)L.o * np;
  float* x_lo = x_hi + (size_t)L.n * op;
  {
    const int64_t total = (int64_t)L.o * L.n;
    const unsigned blocks = (unsigned)std::min<int64_t>(cdiv(total, 256), 4 * kNumSMs);
    gradhat_pack_kernel<<<blocks, 256, 0, st>>>(gw, ldgw, gb, L.o, L.d_in, L.n, np, g_hi, g_lo);
    count_launch();
    if (kfac_status e = check_launch()) return e;
  }
  TcOperand Ainv{h->at<float>(L.Ainv_hi), h->at<float>(L.Ainv_lo), L.n, np};
  TcOperand G{g_hi, g_lo, L.o, np};
  TcEpilogue e1{};
  e1.out_hi = x_hi;
  e1.out_lo = x_lo;
  e1.ldo = op;
  if (kfac_status e = launch_gemm_tc(h, layer, false, TC_EPI_SPLIT, Ainv, G, false, false, L.n,
                                     L.o, L.n, e1, st))
    return e;
  TcOperand Ginv{h->at<float>(L.Ginv_hi), h->at<float>(L.Ginv_lo), L.o, op};
  TcOperand XT{x_hi, x_lo, L.n, op};
  TcEpilogue e2{};
  e2.d_in = L.d_in;
  e2.eta = (float)h->hp.lr;
  e2.mu = (float)h->hp.momentum;
  e2.lambda = (float)h->hp.weight_decay;
  e2.ow = ow;
  e2.ob = ob;
  e2.pw = pw;
  e2.pb = pb;
  e2.mw = h->at<float>(L.m);
  e2.mb = e2.mw + (size_t)L.o * L.d_in;
  return launch_gemm_tc(h, layer, false, TC_EPI_PRECOND, Ginv, XT, false, false, L.o, L.n, L.o,
                        e2, st);
}

}  // namespace kfac
