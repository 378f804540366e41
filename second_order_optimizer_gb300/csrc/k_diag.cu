// K5: diagonal factors   g_new[i] = s sum_r g[r,i]^2,  a_new[j] = s sum_r a[r,j]^2 (+ s*M bias)
// K6: fused diagonal-Fisher step (one streaming pass over the layer's parameters)
//
// "CAFIN: CUDA-accelerated Adaptive Fisher Information Matrix Network
// Optimization via GPU-Native Kernel Fusion", Introduction (AdaFisher keeps
// diagonal Kronecker factors as EMAs) and Kernel Fusion Strategy (one kernel
// loads gradient and parameter into registers, updates the EMA of the diagonal
// Fisher blocks, preconditions, adds momentum and weight decay, and writes the
// parameter in place).  Osawa et al., §5.4: BatchNorm's Fisher is taken as
// diagonal, which is the same step with o = channels, d_in = 1 and a bias.
//
// K6 reads dW, W, m (12 B/param) and writes W, m (8 B/param): 20 B per
// parameter at the HBM roofline.  The per-row and per-column EMA factors are
// recomputed in registers from the old state and the new diagonal; the last
// CTA to finish (a ticket) stores the new EMA vectors, so one launch suffices
// and no CTA ever reads a vector another CTA has already overwritten.
#include "kfac_internal.cuh"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

namespace kfac {

namespace {

constexpr int kDiagThreads = 1024;
constexpr int kK5Threads = 256;
constexpr int64_t kK5MinRows = 32;

// Row splits of K5: enough CTAs for four per SM (rows in flight to cover the HBM
// latency), at least kK5MinRows rows each.
constexpr int kK5CtasPerSm = 4;
int64_t k5_splits(int ncols, int64_t rows) {
  const int64_t cb = cdiv(ncols, kK5Threads);
  int64_t s = cdiv(kK5CtasPerSm * num_sms(), cb);
  s = std::min<int64_t>(s, cdiv(rows, kK5MinRows));
  return std::max<int64_t>(s, 1);
}

struct DiagParams {
  int o, d_in, has_bias;
  float xi, one_minus_xi, gamma, eta, mu, lambda;
  const float* g_new;
  const float* a_new;
  const float* gw;
  const float* gb;
  float* pw;
  float* pb;
  float* ow;
  float* ob;
  float* mw;  // momentum, weight part [o x d_in]
  float* mb;  // momentum, bias part [o]
  float* gs;  // running g diagonal [o]
  float* as;  // running a diagonal [n]
  int* ticket;
};

__device__ __forceinline__ float ema1(float xi, float omx, float old, float nw) {
  return fmaf(xi, old, omx * nw);
}

// One parameter: returns the new W, updates m, optionally stores P.
__device__ __forceinline__ void diag_elem(const DiagParams& p, float gsi, float asj, float gw,
                                          float& w, float& m, float* pout) {
  const float pr = gw / fmaf(gsi, asj, p.gamma);
  const float u = fmaf(p.lambda, w, pr);
  m = fmaf(p.mu, m, u);
  w = fmaf(-p.eta, m, w);
  if (pout) *pout = pr;
}

// Unit u of one layer: VEC: four consecutive weights (u < o d_in / 4), else one
// weight; the last o units are the bias column j = d_in.
template <bool VEC>
__device__ __forceinline__ void diag_unit(const DiagParams& p, int64_t u) {
  const int64_t nw = (int64_t)p.o * p.d_in;
  const int64_t units = VEC ? nw / 4 : nw;
  if (u < units) {
    if (VEC) {
      const int64_t e = u * 4;
      const int i = (int)(e / p.d_in), j = (int)(e % p.d_in);
      const float gsi = ema1(p.xi, p.one_minus_xi, __ldg(p.gs + i), __ldg(p.g_new + i));
      const float4 as4 = __ldg(reinterpret_cast<const float4*>(p.as + j));
      const float4 an4 = __ldg(reinterpret_cast<const float4*>(p.a_new + j));
      const float4 g4 = __ldcs(reinterpret_cast<const float4*>(p.gw + e));
      float4 w4 = __ldcs(reinterpret_cast<const float4*>(p.pw + e));
      float4 m4 = __ldcs(reinterpret_cast<const float4*>(p.mw + e));
      float4 p4;
      diag_elem(p, gsi, ema1(p.xi, p.one_minus_xi, as4.x, an4.x), g4.x, w4.x, m4.x, &p4.x);
      diag_elem(p, gsi, ema1(p.xi, p.one_minus_xi, as4.y, an4.y), g4.y, w4.y, m4.y, &p4.y);
      diag_elem(p, gsi, ema1(p.xi, p.one_minus_xi, as4.z, an4.z), g4.z, w4.z, m4.z, &p4.z);
      diag_elem(p, gsi, ema1(p.xi, p.one_minus_xi, as4.w, an4.w), g4.w, w4.w, m4.w, &p4.w);
      __stcs(reinterpret_cast<float4*>(p.pw + e), w4);
      __stcs(reinterpret_cast<float4*>(p.mw + e), m4);
      if (p.ow) __stcs(reinterpret_cast<float4*>(p.ow + e), p4);
    } else {
      const int i = (int)(u / p.d_in), j = (int)(u % p.d_in);
      const float gsi = ema1(p.xi, p.one_minus_xi, p.gs[i], p.g_new[i]);
      const float asj = ema1(p.xi, p.one_minus_xi, p.as[j], p.a_new[j]);
      float w = p.pw[u], m = p.mw[u];
      diag_elem(p, gsi, asj, p.gw[u], w, m, p.ow ? p.ow + u : nullptr);
      p.pw[u] = w;
      p.mw[u] = m;
    }
  } else {  // bias column j = d_in
    const int i = (int)(u - units);
    const float gsi = ema1(p.xi, p.one_minus_xi, p.gs[i], p.g_new[i]);
    const float asj = ema1(p.xi, p.one_minus_xi, p.as[p.d_in], p.a_new[p.d_in]);
    float w = p.pb[i], m = p.mb[i];
    diag_elem(p, gsi, asj, p.gb[i], w, m, p.ob ? p.ob + i : nullptr);
    p.pb[i] = w;
    p.mb[i] = m;
  }
}

__device__ __forceinline__ int64_t diag_units(const DiagParams& p, bool vec) {
  const int64_t nw = (int64_t)p.o * p.d_in;
  return (vec ? nw / 4 : nw) + (p.has_bias ? p.o : 0);
}

// The new EMA vectors of one layer (called by the last CTA only).
__device__ void diag_store_ema(const DiagParams& p) {
  for (int i = threadIdx.x; i < p.o; i += blockDim.x)
    p.gs[i] = ema1(p.xi, p.one_minus_xi, __ldcg(p.gs + i), p.g_new[i]);
  const int n = p.d_in + p.has_bias;
  for (int j = threadIdx.x; j < n; j += blockDim.x)
    p.as[j] = ema1(p.xi, p.one_minus_xi, __ldcg(p.as + j), p.a_new[j]);
}

// True in every thread of the last CTA to finish (every other CTA has finished
// reading the old EMA vectors); that CTA also resets the ticket.
__device__ __forceinline__ bool last_cta(int* ticket) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  return true;
}

template <bool VEC>
__global__ void __launch_bounds__(kDiagThreads) diag_step_kernel(DiagParams p) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = diag_units(p, VEC);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += stride)
    diag_unit<VEC>(p, u);
  if (!last_cta(p.ticket)) return;
  diag_store_ema(p);
  if (threadIdx.x == 0) *p.ticket = 0;
}

// Several layers in one launch: the layers' units are concatenated (job q owns
// global units [start[q], start[q+1])); a thread walks its units in increasing
// order and reloads the job only when it crosses into the next one.
constexpr int kMaxDiagGroup = 64;
struct DiagGroup {
  DiagParams job[kMaxDiagGroup];
  int64_t start[kMaxDiagGroup + 1];
  int vec[kMaxDiagGroup];
  int count;
  int* ticket;
};

__global__ void __launch_bounds__(kDiagThreads)
diag_step_grouped_kernel(const __grid_constant__ DiagGroup g) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = g.start[g.count];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int q = -1;
  int64_t qbeg = 0, qend = 0;
  int vec = 0;
  DiagParams P{};
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += stride) {
    if (u >= qend) {
      do ++q; while (u >= g.start[q + 1]);
      P = g.job[q];   // by value: registers, not parameter-space reloads
      qbeg = g.start[q];
      qend = g.start[q + 1];
      vec = g.vec[q];
    }
    if (vec) diag_unit<true>(P, u - qbeg);
    else diag_unit<false>(P, u - qbeg);
  }
  if (!last_cta(g.ticket)) return;
  for (int q2 = 0; q2 < g.count; ++q2) diag_store_ema(g.job[q2]);
  if (threadIdx.x == 0) *g.ticket = 0;
}

// K5 ------------------------------------------------------------------------
struct DiagFactorParams {
  const void* a;
  const void* g;
  int64_t lda, ldg, rows, rows_per_split;
  int d_in, o, has_bias, splits, col_blocks;
  float s;
  float* part;     // [splits][d_in + o]
  int* tickets;    // [col_blocks]
  float* g_new;
  float* a_new;
  int vec;         // rows of a and g 16-byte aligned, d_in and o whole 16-byte groups
};

// Squares of this CTA's rows [r0, r1) summed per column, with 16-byte loads:
// thread (tx, ty) owns the 16 / sizeof(T) adjacent columns at tx and the rows
// r0 + ty, r0 + ty + RG, ... (RG row groups), so each warp reads whole row
// segments; eight rows' loads are in flight per thread (eight times the bytes of
// the one-column form).  Each column's RG partials are then added in row-group
// order through shared memory: column cb * 256 + threadIdx.x of the result.
template <typename T>
__device__ __forceinline__ float diag_colsum_vec(const DiagFactorParams& p, int cb, int64_t r0,
                                                 int64_t r1) {
  constexpr int V = 16 / (int)sizeof(T);      // columns per thread
  constexpr int TPR = kK5Threads / V;         // threads across the 256-column block
  constexpr int RG = kK5Threads / TPR;        // row groups
  constexpr int B = 8;                        // rows per batch of loads
  __shared__ float red[RG][kK5Threads];
  const int tx = threadIdx.x % TPR, ty = threadIdx.x / TPR;
  const int c0 = cb * kK5Threads + tx * V;
  float acc[V], comp[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = comp[e] = 0.f;
  auto add = [&](const uint4& w) {
    float x[V];
    if constexpr (sizeof(T) == 2) {
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[2 * h] = __uint_as_float(u[h] << 16);            // lower address
        x[2 * h + 1] = __uint_as_float(u[h] & 0xffff0000u);
      }
    } else {
      x[0] = __uint_as_float(w.x);
      x[1] = __uint_as_float(w.y);
      x[2] = __uint_as_float(w.z);
      x[3] = __uint_as_float(w.w);
    }
#pragma unroll
    for (int e = 0; e < V; ++e) {   // compensated (Kahan) sum per column
      const float y = fmaf(x[e], x[e], -comp[e]);
      const float t = acc[e] + y;
      comp[e] = (t - acc[e]) - y;
      acc[e] = t;
    }
  };
  if (c0 < p.d_in + p.o) {
    const T* base = c0 < p.d_in ? static_cast<const T*>(p.a) + c0
                                : static_cast<const T*>(p.g) + (c0 - p.d_in);
    const int64_t ld = c0 < p.d_in ? p.lda : p.ldg;
    int64_t r = r0 + ty;
    for (; r + (int64_t)(B - 1) * RG < r1; r += (int64_t)B * RG) {
      uint4 w[B];
#pragma unroll
      for (int u = 0; u < B; ++u)
        w[u] = __ldg(reinterpret_cast<const uint4*>(base + (r + (int64_t)u * RG) * ld));
#pragma unroll
      for (int u = 0; u < B; ++u) add(w[u]);
    }
    for (; r < r1; r += RG) add(__ldg(reinterpret_cast<const uint4*>(base + r * ld)));
  }
#pragma unroll
  for (int e = 0; e < V; ++e) red[ty][tx * V + e] = acc[e];
  __syncthreads();
  float v = 0.f;
#pragma unroll
  for (int y = 0; y < RG; ++y) v += red[y][threadIdx.x];
  return v;
}

template <typename T>
__device__ __forceinline__ void diag_factor_body(const DiagFactorParams& p, int cb, int split) {
  const int c = cb * kK5Threads + threadIdx.x;   // 0..d_in-1: a columns; d_in..: g columns
  const int ncols = p.d_in + p.o;
  const int64_t r0 = (int64_t)split * p.rows_per_split;
  const int64_t r1 = min(p.rows, r0 + p.rows_per_split);
  if (p.vec) {
    const float v = diag_colsum_vec<T>(p, cb, r0, r1);
    if (c < ncols) p.part[(size_t)split * ncols + c] = v;
  } else if (c < ncols) {
    const T* base = c < p.d_in ? static_cast<const T*>(p.a) + c
                               : static_cast<const T*>(p.g) + (c - p.d_in);
    const int64_t ld = c < p.d_in ? p.lda : p.ldg;
    // compensated (Kahan) sum: the kernel is bound by HBM, the extra flops are free.
    // Rows in batches of 16: the loads of a batch are independent and issue
    // together; the compensated adds then run in row order.
    float acc = 0.f, comp = 0.f;
    auto kahan = [&](float v) {
      const float y = fmaf(v, v, -comp);
      const float t = acc + y;
      comp = (t - acc) - y;
      acc = t;
    };
    int64_t r = r0;
    for (; r + 16 <= r1; r += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = to_f32<T>(base[(r + u) * ld]);
#pragma unroll
      for (int u = 0; u < 16; ++u) kahan(v[u]);
    }
    for (; r < r1; ++r) kahan(to_f32<T>(base[r * ld]));
    p.part[(size_t)split * ncols + c] = acc;
  }
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(p.tickets + cb, 1) == p.splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (c < ncols) {
    float v = 0.f, comp = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float y = __ldcg(p.part + (size_t)s * ncols + c) - comp;
      const float t = v + y;
      comp = (t - v) - y;
      v = t;
    }
    v *= p.s;
    if (c < p.d_in) p.a_new[c] = v;
    else p.g_new[c - p.d_in] = v;
  }
  if (cb == 0 && threadIdx.x == 0 && p.has_bias) p.a_new[p.d_in] = p.s * (float)p.rows;
  if (threadIdx.x == 0) p.tickets[cb] = 0;
}

template <typename T>
__global__ void __launch_bounds__(kK5Threads) diag_factor_kernel(DiagFactorParams p) {
  pdl_wait();
  pdl_trigger();
  diag_factor_body<T>(p, blockIdx.x, blockIdx.y);
}

// Several layers in one launch: job q owns blocks [block_start[q], block_start[q+1]),
// laid out split-major over its column blocks, with its own partials and tickets.
constexpr int kMaxK5Group = 64;
struct DiagFactorGroup {
  DiagFactorParams job[kMaxK5Group];
  int block_start[kMaxK5Group + 1];
  int count;
};

template <typename T>
__global__ void __launch_bounds__(kK5Threads)
diag_factor_grouped_kernel(const __grid_constant__ DiagFactorGroup g) {
  pdl_wait();
  pdl_trigger();
  int q = 0;
  while (q + 1 < g.count && (int)blockIdx.x >= g.block_start[q + 1]) ++q;
  const DiagFactorParams J = g.job[q];
  const int lb = (int)blockIdx.x - g.block_start[q];
  diag_factor_body<T>(J, lb % J.col_blocks, lb / J.col_blocks);
}

}  // namespace

size_t k5_scratch_floats(int n_plus_o, int64_t max_rows) {
  return (size_t)k5_splits(n_plus_o, max_rows) * (size_t)n_plus_o;
}

namespace {

// K5's 16-byte-load form applies: both inputs' rows start on 16-byte boundaries
// and d_in and o are whole 16-byte groups (no group straddles a and g or passes
// a row's end)
int k5_vec(const void* a, int64_t lda, const void* g, int64_t ldg, int d_in, int o, size_t elt) {
  const int64_t V = 16 / (int64_t)elt;
  auto al16 = [](const void* q) { return q && ((uintptr_t)q & 15) == 0; };
  return al16(a) && al16(g) && lda % V == 0 && ldg % V == 0 && d_in % V == 0 && o % V == 0;
}

DiagFactorParams k5_params(const LayerInfo& L, const void* a, int64_t lda, const void* g,
                           int64_t ldg, int64_t rows, double scale, float* g_new, float* a_new,
                           int64_t splits, float* part, int* tickets) {
  DiagFactorParams p{};
  p.a = a;
  p.g = g;
  p.lda = lda;
  p.ldg = ldg;
  p.rows = rows;
  p.rows_per_split = cdiv(rows, splits);
  p.splits = (int)cdiv(rows, p.rows_per_split);
  p.d_in = L.d_in;
  p.o = L.o;
  p.has_bias = L.has_bias;
  p.col_blocks = (int)cdiv(L.d_in + L.o, kK5Threads);
  p.s = (float)(scale > 0 ? scale : 1.0 / (double)rows);
  p.part = part;
  p.tickets = tickets;
  p.g_new = g_new;
  p.a_new = a_new;
  p.vec = k5_vec(a, lda, g, ldg, L.d_in, L.o, L.in_dtype == KFAC_BF16 ? 2 : 4);
  return p;
}

DiagParams k6_params(kfac_ctx* h, const LayerInfo& L, float decay, const float* g_new,
                     const float* a_new, const float* gw, const float* gb, float* pw, float* pb,
                     float* ow, float* ob, bool* vec) {
  DiagParams p{};
  p.o = L.o;
  p.d_in = L.d_in;
  p.has_bias = L.has_bias;
  p.xi = decay;
  p.one_minus_xi = 1.f - decay;
  p.gamma = (float)h->hp.damping;
  p.eta = (float)h->hp.lr;
  p.mu = (float)h->hp.momentum;
  p.lambda = (float)h->hp.weight_decay;
  p.g_new = g_new;
  p.a_new = a_new;
  p.gw = gw;
  p.gb = gb;
  p.pw = pw;
  p.pb = pb;
  p.ow = ow;
  p.ob = ob;
  p.mw = h->at<float>(L.m);
  p.mb = p.mw + (size_t)L.o * L.d_in;
  p.gs = h->at<float>(L.gs);
  p.as = h->at<float>(L.as);
  p.ticket = h->at<int>(L.ticket);
  auto al16 = [](const void* q) { return ((uintptr_t)q & 15) == 0; };
  *vec = (L.d_in % 4 == 0) && al16(gw) && al16(pw) && al16(p.mw) && al16(p.as) && al16(a_new) &&
         (ow == nullptr || al16(ow));
  return p;
}

int64_t k6_units(const LayerInfo& L, bool vec) {
  const int64_t nw = (int64_t)L.o * L.d_in;
  return (vec ? nw / 4 : nw) + (L.has_bias ? L.o : 0);
}

unsigned k6_blocks(int64_t units) {
  return (unsigned)std::max<int64_t>(std::min<int64_t>(cdiv(units, kDiagThreads), num_sms()), 1);
}

}  // namespace

kfac_status launch_diag_factors(kfac_ctx* h, int layer, const void* a, int64_t lda,
                                const void* g, int64_t ldg, int64_t rows, double scale,
                                float* g_new, float* a_new, cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  DiagFactorParams p = k5_params(L, a, lda, g, ldg, rows, scale, g_new, a_new,
                                 k5_splits(L.d_in + L.o, rows), h->at<float>(h->off_k5part),
                                 h->at<int>(h->off_k5tickets));
  if ((size_t)p.splits * (L.d_in + L.o) > h->k5part_floats) return KFAC_ERR_WORKSPACE;
  dim3 grid(p.col_blocks, p.splits);
  if (L.in_dtype == KFAC_BF16)
    launch_pdl(diag_factor_kernel<__nv_bfloat16>, dim3(grid), dim3(kK5Threads), 0, st, p);
  else
    launch_pdl(diag_factor_kernel<float>, dim3(grid), dim3(kK5Threads), 0, st, p);
  count_launch();
  return check_launch();
}

// Several layers (one input dtype) per launch.  Row splits are shared out so the
// whole group has about kK5CtasPerSm CTAs per SM; each job gets its own partials and
// tickets; a group is cut where the scratch or the job table is full.
kfac_status launch_diag_factors_batched(kfac_ctx* h, int count, const int* layers,
                                        const void* const* a, const int64_t* lda,
                                        const void* const* g, const int64_t* ldg,
                                        const int64_t* rows, double scale,
                                        float* const* g_new, float* const* a_new,
                                        cudaStream_t st) {
  double work = 0;
  for (int i = 0; i < count; ++i) {
    const LayerInfo& L = h->layers[layers[i]];
    work += (double)rows[i] * (L.d_in + L.o);
  }
  const bool bf16 = h->layers[layers[0]].in_dtype == KFAC_BF16;
  DiagFactorGroup grp;
  std::memset(&grp, 0, sizeof(grp));
  size_t used_part = 0, used_tickets = 0;
  int blocks = 0;
  auto flush = [&]() -> kfac_status {
    if (grp.count == 0) return KFAC_OK;
    grp.block_start[grp.count] = blocks;
    if (bf16)
      launch_pdl(diag_factor_grouped_kernel<__nv_bfloat16>, dim3(blocks), dim3(kK5Threads), 0, st, grp);
    else
      launch_pdl(diag_factor_grouped_kernel<float>, dim3(blocks), dim3(kK5Threads), 0, st, grp);
    count_launch();
    grp.count = 0;
    blocks = 0;
    used_part = used_tickets = 0;
    return check_launch();
  };
  for (int i = 0; i < count; ++i) {
    const LayerInfo& L = h->layers[layers[i]];
    const int ncols = L.d_in + L.o;
    const int64_t cb = cdiv(ncols, kK5Threads);
    const double share = (double)rows[i] * ncols / work;   // of kK5CtasPerSm x SMs CTAs
    int64_t splits = (int64_t)std::ceil((double)kK5CtasPerSm * num_sms() * share / (double)cb);
    splits = std::max<int64_t>(1, std::min<int64_t>(splits, cdiv(rows[i], kK5MinRows)));
    const size_t need = (size_t)splits * ncols;
    if (need > h->k5part_floats || (size_t)cb > h->k5tickets_ints) return KFAC_ERR_WORKSPACE;
    if (grp.count == kMaxK5Group || used_part + need > h->k5part_floats ||
        used_tickets + cb > h->k5tickets_ints)
      if (kfac_status e = flush()) return e;
    DiagFactorParams p = k5_params(L, a[i], lda[i], g[i], ldg[i], rows[i], scale, g_new[i],
                                   a_new[i], splits, h->at<float>(h->off_k5part) + used_part,
                                   h->at<int>(h->off_k5tickets) + used_tickets);
    grp.job[grp.count] = p;
    grp.block_start[grp.count] = blocks;
    blocks += p.col_blocks * p.splits;
    ++grp.count;
    used_part += (size_t)p.splits * ncols;
    used_tickets += (size_t)p.col_blocks;
  }
  return flush();
}

kfac_status launch_diag_step(kfac_ctx* h, int layer, float decay, const float* g_new,
                             const float* a_new, const float* gw, const float* gb, float* pw,
                             float* pb, float* ow, float* ob, cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  bool vec = false;
  DiagParams p = k6_params(h, L, decay, g_new, a_new, gw, gb, pw, pb, ow, ob, &vec);
  const unsigned blocks = k6_blocks(k6_units(L, vec));
  if (vec)
    launch_pdl(diag_step_kernel<true>, dim3(blocks), dim3(kDiagThreads), 0, st, p);
  else
    launch_pdl(diag_step_kernel<false>, dim3(blocks), dim3(kDiagThreads), 0, st, p);
  count_launch();
  return check_launch();
}

// Several DIAG layers per launch (up to 64 per group); the ticket of the group's
// first layer orders the EMA write-back.
kfac_status launch_diag_step_batched(kfac_ctx* h, int count, const int* layers,
                                     const float* decay, const float* const* g_new,
                                     const float* const* a_new, const float* const* gw,
                                     const float* const* gb, float* const* pw,
                                     float* const* pb, float* const* ow, float* const* ob,
                                     cudaStream_t st) {
  DiagGroup grp;
  std::memset(&grp, 0, sizeof(grp));
  int64_t units = 0;
  auto flush = [&]() -> kfac_status {
    if (grp.count == 0) return KFAC_OK;
    grp.start[grp.count] = units;
    launch_pdl(diag_step_grouped_kernel, dim3(k6_blocks(units)), dim3(kDiagThreads), 0, st, grp);
    count_launch();
    grp.count = 0;
    units = 0;
    return check_launch();
  };
  for (int i = 0; i < count; ++i) {
    if (grp.count == kMaxDiagGroup)
      if (kfac_status e = flush()) return e;
    const LayerInfo& L = h->layers[layers[i]];
    bool vec = false;
    grp.job[grp.count] = k6_params(h, L, decay[i], g_new[i], a_new[i], gw[i], gb[i], pw[i],
                                   pb[i], ow[i], ob[i], &vec);
    if (grp.count == 0) grp.ticket = grp.job[0].ticket;
    grp.vec[grp.count] = vec;
    grp.start[grp.count] = units;
    units += k6_units(L, vec);
    ++grp.count;
  }
  return flush();
}

namespace {

// K5 for a 2-D convolution, from its NCHW tensors ------------------------------
// A CTA takes one unit -- an input channel ci (its kh x kw patch columns) or an
// output channel (its G column) -- over one range of images.  For an input
// channel it first sums x[b][ci][y][xx]^2 over its images into a shared image
// S[y][xx] (one pass over the input, coalesced along xx); patch column (i, j)
// is then the sum of S over the tap's window, y = oh*sh - ph + i*dh,
// xx = ow*sw - pw + j*dw for the output positions (oh, ow), in bounds.
// Partials go to [split][column]; the last CTA of the launch (one ticket) adds
// them in split order and writes both vectors.
struct DiagConvParams {
  const void* x;
  const void* gy;
  ConvSrc cs;
  int o, has_bias, imgs_per_split;
  int64_t rows;
  float s;
  float* part;     // [splits][C kh kw + o]
  int* ticket;
  float* g_new;
  float* a_new;
};

constexpr size_t kConvSmemMax = 200 * 1024;   // S of one channel: H W floats

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();   // red may still be read by the previous call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kK5Threads / 32; ++w) t += red[w];   // warps in order
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kK5Threads) diag_conv_kernel(const __grid_constant__ DiagConvParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float S[];
  __shared__ float red[kK5Threads / 32];
  __shared__ int s_last;
  const ConvSrc g = p.cs;
  const int u = blockIdx.x, sp = blockIdx.y, tid = threadIdx.x;
  const int khw = g.kh * g.kw, na = g.C * khw, ncols = na + p.o;
  const int b0 = sp * p.imgs_per_split, b1 = min(g.B, b0 + p.imgs_per_split);
  if (u < g.C) {
    const T* x = static_cast<const T*>(p.x);
    const int hw = g.H * g.W;
    // 4 positions x 4 images per step: 16 independent loads in flight per thread
    for (int q0 = tid; q0 < hw; q0 += 4 * kK5Threads) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      int b = b0;
      for (; b + 4 <= b1; b += 4) {
        float v[4][4];
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int q = q0 + k * kK5Threads;
            v[bb][k] = q < hw ? to_f32<T>(x[((int64_t)(b + bb) * g.C + u) * hw + q]) : 0.f;
          }
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
#pragma unroll
          for (int k = 0; k < 4; ++k) acc[k] = fmaf(v[bb][k], v[bb][k], acc[k]);
      }
      for (; b < b1; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int q = q0 + k * kK5Threads;
          const float v = q < hw ? to_f32<T>(x[((int64_t)b * g.C + u) * hw + q]) : 0.f;
          acc[k] = fmaf(v, v, acc[k]);
        }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (q0 + k * kK5Threads < hw) S[q0 + k * kK5Threads] = acc[k];
    }
    __syncthreads();
    const int hwo = g.Ho * g.Wo;
    for (int t = 0; t < khw; ++t) {
      const int i = t / g.kw, j = t - i * g.kw;
      float v = 0.f;
      for (int q = tid; q < hwo; q += kK5Threads) {
        const int oh = q / g.Wo, ow = q - oh * g.Wo;
        const int y = oh * g.sh - g.ph + i * g.dh, xx = ow * g.sw - g.pw + j * g.dw;
        if ((unsigned)y < (unsigned)g.H && (unsigned)xx < (unsigned)g.W) v += S[y * g.W + xx];
      }
      v = block_sum(v, red);
      if (tid == 0) p.part[(size_t)sp * ncols + u * khw + t] = v;
    }
  } else {
    const T* gy = static_cast<const T*>(p.gy);
    const int oc = u - g.C;
    const int64_t hwo = (int64_t)g.Ho * g.Wo;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int b = b0; b < b1; ++b) {
      const T* row = gy + ((int64_t)b * p.o + oc) * hwo;
      for (int64_t q0 = tid; q0 < hwo; q0 += 8 * kK5Threads) {   // 8 loads in flight
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int64_t q = q0 + (int64_t)k * kK5Threads;
          w[k] = q < hwo ? to_f32<T>(row[q]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = fmaf(w[k], w[k], acc[k]);
      }
    }
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) v += acc[k];
    v = block_sum(v, red);
    if (tid == 0) p.part[(size_t)sp * ncols + na + oc] = v;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.ticket, 1) == (int)(gridDim.x * gridDim.y) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int c = tid; c < ncols; c += kK5Threads) {
    float v = 0.f;
    for (int q = 0; q < (int)gridDim.y; ++q) v += __ldcg(p.part + (size_t)q * ncols + c);
    v *= p.s;
    if (c < na) p.a_new[c] = v;
    else p.g_new[c - na] = v;
  }
  if (tid == 0) {
    if (p.has_bias) p.a_new[na] = p.s * (float)p.rows;
    *p.ticket = 0;
  }
}

template <typename T>
bool conv_smem_attr() {
  static bool ok = cudaFuncSetAttribute(diag_conv_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kConvSmemMax) == cudaSuccess;
  return ok;
}

}  // namespace

kfac_status launch_diag_factors_conv(kfac_ctx* h, int layer, const void* x, const void* gy,
                                     const kfac_conv2d_geom& cg, double scale, float* g_new,
                                     float* a_new, cudaStream_t st) {
  const LayerInfo& L = h->layers[layer];
  DiagConvParams p{};
  const int ho = conv_out(cg.in_h, cg.kernel_h, cg.stride_h, cg.pad_h, cg.dilation_h);
  const int wo = conv_out(cg.in_w, cg.kernel_w, cg.stride_w, cg.pad_w, cg.dilation_w);
  p.cs = ConvSrc{cg.batch, cg.in_channels, cg.in_h, cg.in_w, cg.kernel_h, cg.kernel_w,
                 cg.stride_h, cg.stride_w, cg.pad_h, cg.pad_w, cg.dilation_h, cg.dilation_w,
                 ho, wo};
  p.x = x;
  p.gy = gy;
  p.o = L.o;
  p.has_bias = L.has_bias;
  p.rows = (int64_t)cg.batch * ho * wo;
  p.s = (float)(scale > 0 ? scale : 1.0 / (double)p.rows);
  p.g_new = g_new;
  p.a_new = a_new;
  const int units = cg.in_channels + L.o;
  const int64_t ncols = (int64_t)L.d_in + L.o;
  // image splits: about 4096 elements of a unit per CTA (16 loads per thread),
  // and at least two CTAs per SM
  const int64_t per_img = std::max<int64_t>((int64_t)cg.in_h * cg.in_w, (int64_t)ho * wo);
  int64_t splits = std::max<int64_t>(cdiv(2 * num_sms(), units), cdiv(cg.batch * per_img, 4096));
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, cg.batch));
  splits = std::max<int64_t>(1, std::min<int64_t>(splits, (int64_t)(h->k5part_floats / ncols)));
  p.imgs_per_split = (int)cdiv(cg.batch, splits);
  splits = cdiv(cg.batch, p.imgs_per_split);
  if (splits * ncols > (int64_t)h->k5part_floats) return KFAC_ERR_WORKSPACE;
  p.part = h->at<float>(h->off_k5part);
  p.ticket = h->at<int>(h->off_k5tickets);
  const size_t smem = (size_t)cg.in_h * cg.in_w * sizeof(float);
  if (smem > kConvSmemMax) return KFAC_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)units, (unsigned)splits);
  if (L.in_dtype == KFAC_BF16) {
    if (!conv_smem_attr<__nv_bfloat16>()) return KFAC_ERR_CUDA;
    launch_pdl(diag_conv_kernel<__nv_bfloat16>, grid, dim3(kK5Threads), smem, st, p);
  } else {
    if (!conv_smem_attr<float>()) return KFAC_ERR_CUDA;
    launch_pdl(diag_conv_kernel<float>, grid, dim3(kK5Threads), smem, st, p);
  }
  count_launch();
  return check_launch();
}

}  // namespace kfac

// ---------------------------------------------------------------------------
// Workspace-free variant of K5 for callers that cannot allocate device memory.
//
// Some embedders cannot call cudaMalloc or hand the library a workspace: code
// running inside another framework's allocator-controlled region, a plugin
// host that owns every device allocation, or a process that must not grow its
// device footprint after start-up.  For them the scratch of this one kernel
// (row-split partial sums and per-column-block tickets) lives in file-scope
// device arrays that every GPU loading the library holds until process exit.
namespace kfac {
namespace {

constexpr int kStaticMaxCols = 262144;                  // d_in + d_out limit
constexpr int kStaticMaxColBlocks = kStaticMaxCols / kK5Threads;   // 1024
// splits * cols <= ceil(2 SMs / blocks) * blocks * 256 <= 2 SMs * 256 + cols (SMs <= kMaxSMs)
constexpr size_t kStaticScratchFloats = 2 * kMaxSMs * kK5Threads + kStaticMaxCols;

static __device__ __align__(256) float g_k5_static_part[kStaticScratchFloats];
static __device__ __align__(256) int g_k5_static_tickets[kStaticMaxColBlocks];

// Device addresses of the static arrays on the current device.  The names above
// are host-side stand-ins, not device addresses; the lookup is a cheap host call,
// made on every call so that no address outlives the context it came from.
kfac_status static_scratch(float** part, int** tickets) {
  void* p = nullptr;
  void* t = nullptr;
  if (cudaGetSymbolAddress(&p, g_k5_static_part) != cudaSuccess) return KFAC_ERR_CUDA;
  if (cudaGetSymbolAddress(&t, g_k5_static_tickets) != cudaSuccess) return KFAC_ERR_CUDA;
  *part = static_cast<float*>(p);
  *tickets = static_cast<int*>(t);
  return KFAC_OK;
}

}  // namespace
}  // namespace kfac

extern "C" kfac_status kfac_diag_factors_static(const void* a, int64_t lda, const void* g,
                                                int64_t ldg, int64_t rows, int d_in, int d_out,
                                                int has_bias, int in_dtype, double scale,
                                                float* g_new, float* a_new, cudaStream_t stream) {
  using namespace kfac;
  if (!a || !g || !g_new || !a_new) return KFAC_ERR_INVALID_ARG;
  if (d_in < 1 || d_out < 1 || (has_bias != 0 && has_bias != 1)) return KFAC_ERR_INVALID_ARG;
  if (in_dtype != KFAC_F32 && in_dtype != KFAC_BF16) return KFAC_ERR_INVALID_ARG;
  if (rows < 1 || lda < d_in || ldg < d_out || !(scale == scale)) return KFAC_ERR_INVALID_ARG;
  const size_t es = in_dtype == KFAC_BF16 ? 2 : 4;
  if ((uintptr_t)a % es || (uintptr_t)g % es || (uintptr_t)g_new % 4 || (uintptr_t)a_new % 4)
    return KFAC_ERR_INVALID_ARG;
  if ((int64_t)d_in + d_out > kStaticMaxCols) return KFAC_ERR_WORKSPACE;
  float* part = nullptr;
  int* tickets = nullptr;
  if (kfac_status e = static_scratch(&part, &tickets)) return e;
  DiagFactorParams p{};
  p.a = a;
  p.g = g;
  p.lda = lda;
  p.ldg = ldg;
  p.rows = rows;
  const int ncols = d_in + d_out;
  // the row splits as the handle's K5 has them, within what the static array holds
  const int64_t sp = std::max<int64_t>(
      1, std::min<int64_t>(k5_splits(ncols, rows), (int64_t)(kStaticScratchFloats / ncols)));
  p.rows_per_split = cdiv(rows, sp);
  p.splits = (int)cdiv(rows, p.rows_per_split);
  p.d_in = d_in;
  p.o = d_out;
  p.has_bias = has_bias;
  p.col_blocks = (int)cdiv(ncols, kK5Threads);
  p.s = (float)(scale > 0 ? scale : 1.0 / (double)rows);
  p.part = part;
  p.tickets = tickets;
  p.g_new = g_new;
  p.a_new = a_new;
  p.vec = k5_vec(a, lda, g, ldg, d_in, d_out, es);
  if ((size_t)p.splits * ncols > kStaticScratchFloats) return KFAC_ERR_WORKSPACE;
  // the tickets must start at zero; a call interrupted earlier may have left them dirty
  if (cudaMemsetAsync(tickets, 0, sizeof(int) * p.col_blocks, stream) != cudaSuccess)
    return KFAC_ERR_CUDA;
  dim3 grid(p.col_blocks, p.splits);
  if (in_dtype == KFAC_BF16)
    diag_factor_kernel<__nv_bfloat16><<<grid, kK5Threads, 0, stream>>>(p);
  else
    diag_factor_kernel<float><<<grid, kK5Threads, 0, stream>>>(p);
  count_launch();
  return check_launch();
}
