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
// Two products: X = dW-hat . Ainv  ([o x n] . [n x n]) into scratch, then
// P = Ginv . X ([o x o] . [o x n]) whose epilogue writes P and/or updates W, m.
// The bias gradient is read as the virtual last column of dW-hat.
#include "kfac_internal.cuh"
#include "simt_gemm.cuh"

namespace kfac {

namespace {

using KTile = SimtTile<64, 64, 16, 4, 4>;

struct GradHatLoader {  // (i, j) -> [dW | db][i][j]
  const float* gw;
  const float* gb;
  int64_t ld;
  int o, d_in, n;
  __device__ __forceinline__ float operator()(long long i, long long j) const {
    if (i >= o || j >= n) return 0.f;
    if (j < d_in) return gw[i * ld + j];
    return gb[i];
  }
};

__global__ void __launch_bounds__(256) precond_x_kernel(GradHatLoader gh, const float* Ainv,
                                                        float* X) {
  __shared__ float smem[KTile::kSmemFloats];
  const int n = gh.n;
  const int64_t m0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
  float acc[4][4] = {};
  StridedLoader lb{Ainv, n, 1, n, n};
  KTile::run(gh, lb, m0, c0, 0, n, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = m0 + KTile::row_of(i), c = c0 + KTile::col_of(j);
      if (r < gh.o && c < n) X[r * n + c] = acc[i][j];
    }
}

struct UpdateParams {
  int o, d_in, n;
  float eta, mu, lambda;
  float* ow;
  float* ob;
  float* pw;
  float* pb;
  float* mw;
  float* mb;
};

__global__ void __launch_bounds__(256) precond_p_kernel(const float* Ginv, const float* X,
                                                        UpdateParams u) {
  __shared__ float smem[KTile::kSmemFloats];
  const int n = u.n, o = u.o;
  const int64_t m0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
  float acc[4][4] = {};
  StridedLoader la{Ginv, o, 1, o, o};
  StridedLoader lb{X, n, 1, o, n};
  KTile::run(la, lb, m0, c0, 0, o, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = m0 + KTile::row_of(i), c = c0 + KTile::col_of(j);
      if (r >= o || c >= n) continue;
      const float p = acc[i][j];
      if (c < u.d_in) {
        const int64_t e = r * u.d_in + c;
        if (u.ow) u.ow[e] = p;
        if (u.pw) {
          float w = u.pw[e];
          const float m = fmaf(u.mu, u.mw[e], fmaf(u.lambda, w, p));
          u.mw[e] = m;
          u.pw[e] = fmaf(-u.eta, m, w);
        }
      } else {
        if (u.ob) u.ob[r] = p;
        if (u.pb) {
          float w = u.pb[r];
          const float m = fmaf(u.mu, u.mb[r], fmaf(u.lambda, w, p));
          u.mb[r] = m;
          u.pb[r] = fmaf(-u.eta, m, w);
        }
      }
    }
}

}  // namespace

kfac_status launch_precondition(kfac_ctx* h, int layer, const float* gw, int64_t ldgw,
                                const float* gb, float* ow, float* ob, float* pw, float* pb,
                                cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  if ((size_t)L.o * L.n > h->k4tmp_floats) return KFAC_ERR_WORKSPACE;
  float* X = h->at<float>(h->off_k4tmp);
  GradHatLoader gh{gw, gb, ldgw, L.o, L.d_in, L.n};
  dim3 grid((unsigned)cdiv(L.n, 64), (unsigned)cdiv(L.o, 64));
  precond_x_kernel<<<grid, 256, 0, st>>>(gh, h->at<float>(L.Ainv), X);
  count_launch();
  if (kfac_status e = check_launch()) return e;
  UpdateParams u{};
  u.o = L.o;
  u.d_in = L.d_in;
  u.n = L.n;
  u.eta = (float)h->hp.lr;
  u.mu = (float)h->hp.momentum;
  u.lambda = (float)h->hp.weight_decay;
  u.ow = ow;
  u.ob = ob;
  u.pw = pw;
  u.pb = pb;
  u.mw = h->at<float>(L.m);
  u.mb = u.mw + (size_t)L.o * L.d_in;
  precond_p_kernel<<<grid, 256, 0, st>>>(h->at<float>(L.Ginv), X, u);
  count_launch();
  return check_launch();
}

}  // namespace kfac
