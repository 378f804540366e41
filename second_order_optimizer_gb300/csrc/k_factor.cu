// K1: running Kronecker factors  F <- beta F + alpha x-hat^T x-hat  (upper triangle + mirror).
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", §3.2 (A from the layer's input
// activations, G from its output gradients) and §3.4 (a symmetric factor has
// N(N+1)/2 distinct entries: only tiles on or above the diagonal are computed,
// the epilogue writes each entry and its mirror).  The EMA of the CAFIN
// briefing (Introduction) is the epilogue's beta*F_old + alpha*acc with
// alpha = (1-xi) s, beta = xi.
//
// This translation unit holds the CUDA-core (FP32 FFMA) grouped SYRK used for
// the inverse assembly Finv = X^T X and, for the factor update, whenever the
// tensor-core path does not apply.  Split-K partial tiles are reduced by the
// last CTA of each tile (a per-tile ticket), in fixed split order, so the
// result is deterministic and no separate reduction launch is needed.
#include "kfac_internal.cuh"
#include "simt_gemm.cuh"
#include "syrk_simt.cuh"

#include <algorithm>
#include <vector>

namespace kfac {

namespace {

template <typename T>
struct XhatLoader {  // (col, row) -> x-hat[row][col]
  const T* x;
  int64_t ld, M;
  int d, n;
  __device__ __forceinline__ float operator()(long long col, long long row) const {
    if (row >= M || col >= n) return 0.f;
    if (col >= d) return 1.f;  // the ones column (only present when n > d)
    return to_f32<T>(x[row * ld + col]);
  }
};
template <typename T>
struct XhatLoaderT {  // (row, col) -> x-hat[row][col]
  XhatLoader<T> l;
  __device__ __forceinline__ float operator()(long long row, long long col) const {
    return l(col, row);
  }
};

__device__ __forceinline__ void tile_coords(int t, int nt, int* ti, int* tj) {
  int r = 0;
  while (t >= nt - r) {
    t -= nt - r;
    ++r;
  }
  *ti = r;
  *tj = r + t;
}

__device__ __forceinline__ void syrk_store(const SyrkJob& j, int64_t gr, int64_t gc, float acc) {
  if (gr >= j.n || gc >= j.n || gr > gc) return;
  float* p = j.C + gr * j.n + gc;
  float v = j.alpha * acc;
  if (j.beta != 0.f) v = fmaf(j.beta, *p, v);
  *p = v;
  if (gr != gc) j.C[gc * j.n + gr] = v;
}

template <typename T>
__global__ void __launch_bounds__(SyrkTile::Tile::kThreads)
syrk_simt_kernel(const SyrkJob* __restrict__ jobs, SyrkJob job0) {
  pdl_wait();
  pdl_trigger();
  using Tile = SyrkTile::Tile;
  constexpr int BM = SyrkTile::BM, BN = SyrkTile::BN, TM = SyrkTile::TM, TN = SyrkTile::TN;
  __shared__ float smem[Tile::kSmemFloats];
  __shared__ int s_last;
  const SyrkJob j = jobs ? jobs[blockIdx.y] : job0;
  if (j.skip) return;
  const int tiles = j.nt * (j.nt + 1) / 2;
  if ((int)blockIdx.x >= tiles * j.splits) return;
  const int tile = blockIdx.x / j.splits, split = blockIdx.x % j.splits;
  int ti, tj;
  tile_coords(tile, j.nt, &ti, &tj);
  int64_t r0 = (int64_t)split * j.rows_per_split;
  int64_t r1 = min(j.M, r0 + j.rows_per_split);
  if (j.x_lower) r0 = max(r0, (int64_t)tj * BN);  // x[r][c] = 0 for r < c
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int k = 0; k < TN; ++k) acc[i][k] = 0.f;
  XhatLoader<T> la{static_cast<const T*>(j.x), j.ld, j.M, j.d, j.n};
  XhatLoaderT<T> lb{la};
  if (r0 < r1) Tile::run(la, lb, (long long)ti * BM, (long long)tj * BN, r0, r1, acc, smem);

  if (j.splits == 1) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int k = 0; k < TN; ++k)
        syrk_store(j, (int64_t)ti * BM + Tile::row_of(i), (int64_t)tj * BN + Tile::col_of(k),
                   acc[i][k]);
    return;
  }
  float* part = j.part + (size_t)tile * j.splits * (BM * BN);
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int k = 0; k < TN; ++k)
      part[(size_t)split * (BM * BN) + Tile::row_of(i) * BN + Tile::col_of(k)] = acc[i][k];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&j.tickets[tile], 1) == j.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int k = 0; k < TN; ++k) {
      const int e = Tile::row_of(i) * BN + Tile::col_of(k);
      float v = 0.f;
      for (int s = 0; s < j.splits; ++s) v += __ldcg(part + (size_t)s * (BM * BN) + e);
      syrk_store(j, (int64_t)ti * BM + Tile::row_of(i), (int64_t)tj * BN + Tile::col_of(k), v);
    }
  if (threadIdx.x == 0) j.tickets[tile] = 0;
}

}  // namespace

kfac_status launch_syrk_simt(const SyrkJob* job, int njobs, bool bf16, cudaStream_t st) {
  if (njobs != 1) return KFAC_ERR_INVALID_ARG;
  const int tiles = job->nt * (job->nt + 1) / 2;
  dim3 grid(tiles * job->splits, 1);
  if (bf16)
    launch_pdl(syrk_simt_kernel<__nv_bfloat16>, dim3(grid), dim3(SyrkTile::Tile::kThreads), 0, st, nullptr, *job);
  else
    launch_pdl(syrk_simt_kernel<float>, dim3(grid), dim3(SyrkTile::Tile::kThreads), 0, st, nullptr, *job);
  count_launch();
  return check_launch();
}

kfac_status launch_syrk_simt_grouped(const SyrkJob* d_jobs, int njobs, int max_tiles,
                                     cudaStream_t st) {
  if (njobs <= 0) return KFAC_OK;
  dim3 grid(max_tiles, njobs);
  launch_pdl(syrk_simt_kernel<float>, dim3(grid), dim3(SyrkTile::Tile::kThreads), 0, st, d_jobs, SyrkJob{});
  count_launch();
  return check_launch();
}

namespace {
constexpr int64_t kMaxRowsPerSplit = 8192;
constexpr int64_t kMinRowsPerSplit = 256;
}  // namespace

// Split plan shared by the planner (scratch sizing) and the launcher: enough
// CTAs to fill the GPU twice, at least kMinRowsPerSplit rows per split, and at
// most kMaxRowsPerSplit rows summed by one thread (bounds fp32 error growth).
static int64_t split_count_before_rounding(int n, int64_t rows) {
  int nt = (int)cdiv(n, SyrkTile::BM);
  int64_t tiles = (int64_t)nt * (nt + 1) / 2;
  int64_t s = cdiv(2 * num_sms(), tiles);   // two CTAs per SM
  s = std::min<int64_t>(s, std::max<int64_t>(1, rows / kMinRowsPerSplit));
  s = std::max<int64_t>(s, cdiv(rows, kMaxRowsPerSplit));
  return std::max<int64_t>(s, 1);
}

void syrk_split_plan(int n, int64_t rows, int* splits_out, int64_t* rows_per_split_out) {
  int64_t s = split_count_before_rounding(n, rows);
  int64_t rps = cdiv(cdiv(rows, s), SyrkTile::BK) * SyrkTile::BK;
  *splits_out = (int)cdiv(rows, rps);
  *rows_per_split_out = rps;
}

size_t k1_scratch_floats(int n, int64_t max_rows, size_t* tickets) {
  int nt = (int)cdiv(n, SyrkTile::BM);
  int64_t tiles = (int64_t)nt * (nt + 1) / 2;
  *tickets = (size_t)tiles;
  // the split count never exceeds its value before rounding, which grows with rows
  int64_t s = split_count_before_rounding(n, max_rows);
  return s > 1 ? (size_t)(tiles * s) * SyrkTile::BM * SyrkTile::BN : 0;
}

kfac_status launch_update_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                  const void* g, int64_t ldg, int64_t rows, double scale,
                                  float decay_a, float decay_g, cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  const double s = scale > 0 ? scale : 1.0 / (double)rows;
  const bool bf16 = L.in_dtype == KFAC_BF16;
  if (a) {
    const float alpha = (float)((1.0 - (double)decay_a) * s);
    kfac_status e = launch_syrk_tc(h, layer, a, lda, rows, L.d_in, L.n, L.has_bias, bf16, alpha,
                                   decay_a, h->at<float>(L.A), st);
    if (e != KFAC_OK) return e;
  }
  if (!g) return KFAC_OK;
  const float alpha = (float)((1.0 - (double)decay_g) * s);
  return launch_syrk_tc(h, layer, g, ldg, rows, L.o, L.o, 0, bf16, alpha, decay_g,
                        h->at<float>(L.G), st);
}

// Several layers' factor updates at once: every a and g of a group is packed in
// one launch, then all their SYRKs run as one grouped tensor-core launch (tiles
// of all layers fill the GPU together instead of each layer splitting K).  A
// group is as many layers as the pack scratch holds.  A null a[i] (g[i]) leaves
// that layer's A (G) as it is.
kfac_status launch_update_factors_batched(kfac_ctx* h, int count, const int* layers,
                                          const void* const* a, const int64_t* lda,
                                          const void* const* g, const int64_t* ldg,
                                          const int64_t* rows, double scale,
                                          const float* decay_a, const float* decay_g,
                                          cudaStream_t st, const kfac_conv2d_geom* geoms) {
  const bool bf16 = h->layers[layers[0]].in_dtype == KFAC_BF16;
  const size_t elt = bf16 ? 2 : 8;  // packed bytes per element (bf16, or two TF32 halves)
  std::vector<PackJob> pj;
  std::vector<TcProblem> pr, direct;
  size_t used = 0;
  // bf16 inputs that the CTA-pair SYRK can read in place (launch_syrk_direct) skip
  // the pack, when together they fill at least one wave of CTA pairs
  auto direct_ok = [&](int i, int w) {
    const LayerInfo& L = h->layers[layers[i]];
    const void* src = w == 0 ? a[i] : g[i];
    return bf16 && !geoms && src &&
           syrk_direct_layout_ok(h, src, w == 0 ? lda[i] : ldg[i], rows[i],
                                 w == 0 ? L.d_in : L.o, w == 0 ? L.has_bias : 0);
  };
  int64_t direct_tiles = 0;
  for (int i = 0; i < count; ++i)
    for (int w = 0; w < 2; ++w)
      if (direct_ok(i, w)) direct_tiles += syrk_pair_tiles(w == 0 ? h->layers[layers[i]].n : h->layers[layers[i]].o);
  const bool use_direct = direct_tiles >= num_sms() / 2;
  auto flush = [&]() -> kfac_status {
    if (pr.empty()) return KFAC_OK;
    kfac_status e = launch_pack_grouped(pj.data(), (int)pj.size(), bf16, st);
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, bf16, TC_EPI_SYRK, pr.data(), (int)pr.size(), st);
    pj.clear();
    pr.clear();
    used = 0;
    return e;
  };
  for (int i = 0; i < count; ++i) {
    const LayerInfo& L = h->layers[layers[i]];
    const int64_t Kp = tc_pitch(rows[i], bf16);
    const bool dA = use_direct && direct_ok(i, 0), dG = use_direct && direct_ok(i, 1);
    const size_t bA = a[i] && !dA ? align_up((size_t)L.n * Kp * elt) : 0;
    const size_t bG = g[i] && !dG ? align_up((size_t)L.o * Kp * elt) : 0;
    if (bA + bG > h->tcpack_bytes) return KFAC_ERR_WORKSPACE;
    if (used + bA + bG > h->tcpack_bytes)
      if (kfac_status e = flush()) return e;
    const double s = scale > 0 ? scale : 1.0 / (double)rows[i];
    for (int w = 0; w < 2; ++w) {
      const void* src = w == 0 ? a[i] : g[i];
      if (!src) continue;
      const float decay = w == 0 ? decay_a[i] : decay_g[i];
      const float alpha = (float)((1.0 - (double)decay) * s);
      const int n = w == 0 ? L.n : L.o;
      if (w == 0 ? dA : dG) {
        TcProblem q{};
        q.A = TcOperand{src, nullptr, w == 0 ? L.d_in : L.o, w == 0 ? lda[i] : ldg[i]};
        q.B = q.A;
        q.same_ab = true;
        q.upper = true;
        q.M = q.N = n;
        q.K = rows[i];
        q.bias_col = (w == 0 && L.has_bias) ? L.d_in : -1;
        q.e.alpha = alpha;
        q.e.beta = decay;
        q.e.C = h->at<float>(w == 0 ? L.A : L.G);
        q.e.ldc = n;
        q.layer = layers[i];
        direct.push_back(q);
        continue;
      }
      char* hi = h->ws + h->off_tcpack + used;
      char* lo = bf16 ? nullptr : hi + (size_t)n * Kp * 4;
      used += w == 0 ? bA : bG;
      PackJob j{};
      j.x = src;
      j.ld = geoms ? 0 : (w == 0 ? lda[i] : ldg[i]);
      j.M = rows[i];
      if (geoms) {
        const kfac_conv2d_geom& cg = geoms[i];
        const int ho = conv_out(cg.in_h, cg.kernel_h, cg.stride_h, cg.pad_h, cg.dilation_h);
        const int wo = conv_out(cg.in_w, cg.kernel_w, cg.stride_w, cg.pad_w, cg.dilation_w);
        j.conv = 1;
        if (w == 0)
          j.cs = ConvSrc{cg.batch, cg.in_channels, cg.in_h, cg.in_w, cg.kernel_h, cg.kernel_w,
                         cg.stride_h, cg.stride_w, cg.pad_h, cg.pad_w, cg.dilation_h,
                         cg.dilation_w, ho, wo};
        else  // the output gradient is its own 1x1 unit-stride "input"
          j.cs = ConvSrc{cg.batch, L.o, ho, wo, 1, 1, 1, 1, 0, 0, 1, 1, ho, wo};
      }
      j.d = w == 0 ? L.d_in : L.o;
      j.n = n;
      j.Kp = Kp;
      j.hi = hi;
      j.lo = lo;
      pj.push_back(j);
      TcProblem q{};
      q.A = TcOperand{hi, lo, n, Kp};
      q.B = q.A;
      q.same_ab = true;
      q.upper = true;
      q.M = q.N = n;
      q.K = rows[i];
      q.e.alpha = alpha;
      q.e.beta = decay;
      q.e.C = h->at<float>(w == 0 ? L.A : L.G);
      q.e.ldc = n;
      q.layer = layers[i];
      pr.push_back(q);
    }
  }
  if (kfac_status e = flush()) return e;
  return direct.empty() ? KFAC_OK : launch_syrk_direct(h, direct.data(), (int)direct.size(), st);
}

}  // namespace kfac
