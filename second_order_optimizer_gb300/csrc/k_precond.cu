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
// Both products run on the tensor cores with fp32 operands split as
// v = h + r, h the TF32 rounding: the product of the h's in TF32 plus the two
// cross terms h_a r_b + r_a h_b in one bf16 MMA over bf16 roundings of h and r
// (tc::corr_pair).  That is two MMA issues per 8 k against three for 3xTF32,
// and the dropped parts (r_a r_b, the bf16 rounding of the cross terms) are
// about 2^-20 of each product: P within ~1e-6 of its exact value at
// cond(F) = 2e4 against ~1e-7 for 3xTF32.
//   pack     dW-hat = [dW | db] -> hi [o x n_p] + correction pairs (A form)
//   X    =   dW-hat . Ainv        M = o, N = n, K = n   epilogue stores X^T (hi + A-form pairs)
//   P^T  =   X^T . Ginv           M = n, N = o, K = o   epilogue: P out and/or W, m update
// (Ainv and Ginv are symmetric.)  Storing X^T keeps every operand K-major, and
// with the products oriented this way each epilogue thread, which holds one
// accumulator row, writes to consecutive addresses across a warp.  Ainv/Ginv
// operands (hi + B-form pairs) are produced once per refresh by the inverse pass.
#include "kfac_internal.cuh"
#include "tc_prims.cuh"

#include <algorithm>
#include <cstring>
#include <vector>

namespace kfac {

namespace {

struct GradPackJob {
  const float* gw;
  const float* gb;
  int64_t ld, np;
  int o, d_in, n;
  float* hi;
  float* lo;      // correction pairs (tc::corr_pair, A form); null: bf16 values
                  // in hi, row pitch 2 np elements
  int vec;        // rows of gw, hi and lo 16-byte aligned: float4 over the weight columns
};
constexpr int kMaxGradPack = 16;
struct GradPackGroup {
  GradPackJob job[kMaxGradPack];
};

__global__ void __launch_bounds__(256) gradhat_pack_grouped_kernel(
    const __grid_constant__ GradPackGroup g) {
  pdl_wait();
  pdl_trigger();
  const GradPackJob J = g.job[blockIdx.y];  // by value: no reloads after each store
  // a CTA takes whole rows (no index division), its threads along the row; with
  // J.vec the weight columns go four at a time and the rest (the bias) one by one
  const int j0 = J.vec ? J.d_in / 4 * 4 : 0;
  for (int i = blockIdx.x; i < J.o; i += gridDim.x) {
    const float* src = J.gw + (int64_t)i * J.ld;
    if (!J.lo) {   // bf16 operand
      __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(J.hi) + (int64_t)i * 2 * J.np;
#pragma unroll 2
      for (int j = 4 * threadIdx.x; j < j0; j += 4 * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src + j));
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v.x, v.y), p1 = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(b + j) = u;
      }
#pragma unroll 4
      for (int j = j0 + threadIdx.x; j < J.n; j += blockDim.x)
        b[j] = __float2bfloat16_rn(j < J.d_in ? __ldg(src + j) : J.gb[i]);
      continue;
    }
    // TF32 + bf16-correction form (A operand)
    float* hi = J.hi + (int64_t)i * J.np;
    uint32_t* lo = reinterpret_cast<uint32_t*>(J.lo) + (int64_t)i * J.np;
#pragma unroll 2
    for (int j = 4 * threadIdx.x; j < j0; j += 4 * blockDim.x) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src + j));
      float4 h;
      uint4 l;
      h.x = tc::corr_pair(v.x, false, &l.x);
      h.y = tc::corr_pair(v.y, false, &l.y);
      h.z = tc::corr_pair(v.z, false, &l.z);
      h.w = tc::corr_pair(v.w, false, &l.w);
      *reinterpret_cast<float4*>(hi + j) = h;
      *reinterpret_cast<uint4*>(lo + j) = l;
    }
#pragma unroll 4
    for (int j = j0 + threadIdx.x; j < J.n; j += blockDim.x)
      hi[j] = tc::corr_pair(j < J.d_in ? __ldg(src + j) : J.gb[i], false, &lo[j]);
  }
}

// TMEM drain period of the two 3xTF32 products (k elements): 512 instead of the
// default 128 gives the PRECOND epilogue, whose loads of W and m take longer than
// two 128-k periods of MMAs, room to overlap the next tile (transformer
// preconditioning 12.1 -> 11.5 ms; P of its layers within 2e-5 of float64).  The
// inversion's products keep 128: at cond 2e4 their longer chains doubled the
// inverse's error.
constexpr int kPrecondDrainK = 512;

}  // namespace

kfac_status launch_precondition(kfac_ctx* h, int layer, const float* gw, int64_t ldgw,
                                const float* gb, float* ow, float* ob, float* pw, float* pb,
                                cudaStream_t st) {
  // one layer through the batched path (the products of a group of one layer are
  // single products there)
  return launch_precondition_batched(h, 1, &layer, &gw, &ldgw, &gb, ow ? &ow : nullptr,
                                     ob ? &ob : nullptr, pw ? &pw : nullptr, pb ? &pb : nullptr,
                                     st);
}

// Several layers at once: one pack launch for all gradients, then each of the two
// products as one grouped tensor-core launch over all layers of the group.  A
// group is as many layers as the scratch holds (at most 16).
kfac_status launch_precondition_batched(kfac_ctx* h, int count, const int* layers,
                                        const float* const* gw, const int64_t* ldgw,
                                        const float* const* gb, float* const* ow,
                                        float* const* ob, float* const* pw, float* const* pb,
                                        cudaStream_t st) {
  // bf16 preconditioning: gradients, inverses and X^T as bf16 (row pitch 2 np / 2 op
  // elements, in the storage of the TF32 hi halves), one bf16 product each
  const bool bf = h->hp.math == KFAC_MATH_BF16;
  std::vector<TcProblem> p1, p2;
  GradPackGroup gp;
  std::memset(&gp, 0, sizeof(gp));
  int ng = 0;
  int64_t max_rows = 0;
  size_t used = 0;  // floats
  auto flush = [&]() -> kfac_status {
    if (ng == 0) return KFAC_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(max_rows, 4 * num_sms());
    launch_pdl(gradhat_pack_grouped_kernel, dim3(dim3(blocks, ng)), dim3(256), 0, st, gp);
    count_launch();
    kfac_status e = check_launch();
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, bf, TC_EPI_SPLIT, p1.data(), ng, st);
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, bf, TC_EPI_PRECOND, p2.data(), ng, st);
    p1.clear();
    p2.clear();
    ng = 0;
    max_rows = 0;
    used = 0;
    return e;
  };
  for (int i = 0; i < count; ++i) {
    const LayerInfo& L = h->layers[layers[i]];
    const int64_t np = tc_pitch(L.n, false), op = tc_pitch(L.o, false);
    const size_t gfl = align_up((size_t)L.o * np * 4) / 4, xfl = align_up((size_t)L.n * op * 4) / 4;
    const size_t need = 2 * gfl + 2 * xfl;
    if (need > h->k4tmp_floats) return KFAC_ERR_WORKSPACE;
    if (used + need > h->k4tmp_floats || ng == kMaxGradPack)
      if (kfac_status e = flush()) return e;
    float* g_hi = h->at<float>(h->off_k4tmp) + used;
    float* g_lo = g_hi + gfl;
    float* x_hi = g_lo + gfl;
    float* x_lo = x_hi + xfl;
    used += need;
    GradPackJob& j = gp.job[ng];
    j.gw = gw[i];
    j.gb = gb[i];
    j.ld = ldgw[i];
    j.np = np;
    j.o = L.o;
    j.d_in = L.d_in;
    j.n = L.n;
    j.hi = g_hi;
    j.lo = bf ? nullptr : g_lo;
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    j.vec = ldgw[i] % 4 == 0 && np % 4 == 0 && al16(gw[i]) && al16(g_hi) && (bf || al16(g_lo));
    max_rows = std::max<int64_t>(max_rows, L.o);
    const int64_t npb = bf ? 2 * np : np, opb = bf ? 2 * op : op;   // operand pitches
    TcProblem q1{};
    const int corr = bf ? 0 : 1;
    q1.A = TcOperand{g_hi, bf ? nullptr : g_lo, L.o, npb, corr};   // X = grad-hat . Ainv, as X^T
    q1.B = TcOperand{h->at<float>(L.Ainv_hi), bf ? nullptr : h->at<float>(L.Ainv_lo), L.n, npb,
                     corr};
    q1.M = L.o;
    q1.N = L.n;
    q1.K = L.n;
    q1.e.out_hi = x_hi;
    q1.e.out_lo = bf ? nullptr : x_lo;
    q1.e.out_corr = corr;
    q1.e.out_bf16 = bf ? 1 : 0;
    q1.e.alpha = 1.f;
    q1.e.ldo = opb;
    q1.layer = layers[i];
    q1.drain_k = kPrecondDrainK;
    p1.push_back(q1);
    TcProblem q2{};
    q2.A = TcOperand{x_hi, bf ? nullptr : x_lo, L.n, opb, corr};   // P^T = X^T . Ginv
    q2.B = TcOperand{h->at<float>(L.Ginv_hi), bf ? nullptr : h->at<float>(L.Ginv_lo), L.o, opb,
                     corr};
    q2.M = L.n;
    q2.N = L.o;
    q2.K = L.o;
    q2.e.d_in = L.d_in;
    q2.e.eta = (float)h->hp.lr;
    q2.e.mu = (float)h->hp.momentum;
    q2.e.lambda = (float)h->hp.weight_decay;
    q2.e.ow = ow ? ow[i] : nullptr;
    q2.e.ob = ob ? ob[i] : nullptr;
    q2.e.pw = pw ? pw[i] : nullptr;
    q2.e.pb = pb ? pb[i] : nullptr;
    q2.e.mw = h->at<float>(L.m);
    q2.e.mb = q2.e.mw + (size_t)L.o * L.d_in;
    q2.layer = layers[i];
    q2.drain_k = kPrecondDrainK;
    p2.push_back(q2);
    ++ng;
  }
  return flush();
}

}  // namespace kfac
