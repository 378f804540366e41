// K2 + K3: damped inverses  F_d^{-1} = (F + sqrt(gamma) I)^{-1}  for every factor, batched.
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...", §3.2: the inverse of the
// Kronecker-factored Fisher is taken through the inverses of the two factors;
// §3.3 notes that this inverse work is the main overhead of K-FAC, and §5.4
// that it need not be refreshed every step (the caller decides the cadence).
// The pages give no inversion algorithm; this file uses the standard one for
// symmetric positive-definite matrices:
//
//   1. L = lower(F) + sqrt(gamma) I                                 (prep)
//   2. blocked right-looking Cholesky, block nb = 64, per block column k:
//        diag:     L_kk = chol(L_kk) in shared memory; X_kk = L_kk^{-1}
//        panel:    L_ik <- L_ik L_kk^{-T}                 (i > k)
//        trailing: L_ij <- L_ij - L_ik L_jk^T              (i >= j > k, lower tiles)
//   3. X = L^{-1} by recursive doubling over block pairs:
//        X_BT = -X_BB (L_BT X_TT)        for pairs (T, B) of size s = 64, 128, ...
//   4. F_d^{-1} = X^T X  (grouped SYRK, upper tiles + mirror)
//
// Every matrix of the batch runs the same step sequence; a matrix whose size
// is already exhausted at a step returns at once.  A pivot that is not > 0 (or
// not finite) is reported as KFAC_ERR_NOT_PD with its 0-based column, replaced
// by 1 so the rest of the pass stays finite, and the result is flagged.
#include "kfac_internal.cuh"
#include "simt_gemm.cuh"
#include "syrk_simt.cuh"
#include "tc_prims.cuh"

#include <algorithm>
#include <cstring>
#include <memory>
#include <vector>

namespace kfac {

namespace {

constexpr int NB = 64;
constexpr int kOuterW = 512;      // outer panel width of the blocked Cholesky
constexpr int kMidW = 256;        // half of an outer panel: its second half gets the first on the tensor cores
constexpr int kOuterMaxN = 1536;  // handles whose factors are all this small stay one panel
constexpr int kTcLevelMin = 512;  // doubling levels of this block size and wider: tensor cores
using PTile = SimtTile<64, 64, 32, 4, 4>;   // 256 threads, 32-deep k chunks

__global__ void __launch_bounds__(256) inv_prep_kernel(const InvJob* jobs, float sqrt_gamma) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  // rows over the grid, columns over the threads (no index division per element);
  // both triangles (F is symmetric): the tensor-core trailing updates of large
  // factors read either triangle and keep the trailing block symmetric.  X needs
  // no clearing: every refresh rewrites its lower triangle (diagonal blocks with
  // their zeros above the diagonal, then every block below by the doubling
  // levels), and its strict upper triangle outside the diagonal blocks, zero
  // since kfac_create, is never written.
  for (int r = blockIdx.x; r < J.n; r += gridDim.x) {
    const int64_t row = (int64_t)r * J.n;
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) {
      const float f = J.F[row + c];
      J.L[row + c] = r == c ? f + sqrt_gamma : f;
    }
  }
}

// Diagonal block b x b (b <= 64) at (k, k): L_kk = chol(block) and X_kk = L_kk^{-1}.
// The block sits in shared memory (rows >= b padded with the identity) and is
// factored in 16-column sub-panels:
//   (a) one warp factors the 16 x 16 diagonal sub-block D = L_D L_D^T: lane r
//       holds row r in registers; each column's multipliers reach the other
//       lanes by warp shuffles, so the 16 dependent steps need no block barrier;
//   (b) the rows below become L_below = A_below L_D^{-T}, one thread per row by
//       forward substitution;
//   (c) the trailing lower triangle: A <- A - L_below L_below^T.
// X_kk then follows from its diagonal 1 / L_ii by doubling over block pairs of
// size 1 to 32, X_BT = -X_BB (L_BT X_TT).  A pivot that is not > 0 and finite is
// recorded (first failing column), replaced by 1, and reported once per
// sub-panel.
// (Measured on GB300 with clock stamps: a per-column version that kept the
// whole block in registers of 256 threads paid a block barrier and a
// shared-memory round trip per column, ~1500 cycles a column; forming each D^{-1}
// inside the warp's pivot loop as well, ~420 cycles a column and 42.8k cycles
// for the block; this form ~205 cycles a column and 29.6k for the block.)
constexpr int SB = 16;       // sub-panel width
constexpr int AP = NB + 1;   // shared row pitch (floats)
constexpr unsigned kFull = 0xffffffffu;

// One doubling level of the 64 x 64 block inverse: for the pairs (T, B) of
// size SZ, X_BT = -X_BB (L_BT X_TT).  The triangular operands hold exact zeros
// outside their triangles, so every sum runs over the whole block length (same
// nonzero terms in the same order) with fixed trip counts the compiler unrolls.
template <int SZ>
__device__ __forceinline__ void diag_inverse_level(const float* A, float* X, float* Y, int tid) {
  constexpr int TOT = (NB / (2 * SZ)) * SZ * SZ;   // outputs of the level
  constexpr int PER = (TOT + 255) / 256;           // per thread, at most
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int e = tid + 256 * u;
    if (TOT % 256 != 0 && e >= TOT) break;
    const int pr = e / (SZ * SZ), i = (e / SZ) % SZ, c = e % SZ;
    const int T0 = pr * 2 * SZ, B0 = T0 + SZ;
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < SZ; ++m) acc = fmaf(A[(B0 + i) * AP + T0 + m], X[(T0 + m) * AP + T0 + c], acc);
    Y[(pr * SZ + i) * 33 + c] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int e = tid + 256 * u;
    if (TOT % 256 != 0 && e >= TOT) break;
    const int pr = e / (SZ * SZ), i = (e / SZ) % SZ, c = e % SZ;
    const int T0 = pr * 2 * SZ, B0 = T0 + SZ;
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < SZ; ++m) acc = fmaf(X[(B0 + i) * AP + B0 + m], Y[(pr * SZ + m) * 33 + c], acc);
    X[(B0 + i) * AP + T0 + c] = -acc;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256, 1) chol_diag_kernel(const InvJob* jobs, int k,
                                                        DevStatus* st) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.x];
  if (k >= J.n) return;
  const int b = min(NB, J.n - k);
  const int n = J.n;
  __shared__ float A[NB * AP];
  __shared__ float X[NB * AP];
  __shared__ float Y[32 * 33];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {   // all sixteen loads in flight before the first shared-memory store
    constexpr int U = NB * NB / 256;
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = tid + 256 * u;
      const int r = e / NB, c = e % NB;
      v[u] = (r < b && c <= r) ? J.L[(int64_t)(k + r) * n + k + c] : (r == c ? 1.f : 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = tid + 256 * u;
      const int r = e / NB, c = e % NB;
      A[r * AP + c] = v[u];
      X[r * AP + c] = 0.f;
    }
  }
  __syncthreads();
  for (int p = 0; p < NB / SB; ++p) {
    const int o = p * SB;
    if (warp == 0) {   // (a)
      const int r = lane & (SB - 1);   // lanes 16..31 mirror 0..15
      float s[SB];
#pragma unroll
      for (int c = 0; c < SB; ++c) s[c] = (c <= r) ? A[(o + r) * AP + o + c] : 0.f;
      int bad = -1;
      float rinv = 0.f;   // 1 / L_rr
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        float d = __shfl_sync(kFull, s[j], j);
        const bool ok = d > 0.f && d <= 3.402823466e38f;   // positive and finite
        bad = (!ok && bad < 0) ? j : bad;
        d = ok ? d : 1.f;
        const float inv = rsqrtf(d), sq = d * inv;
        const float l = r > j ? s[j] * inv : 0.f;
        s[j] = r == j ? sq : (r > j ? l : s[j]);
        rinv = r == j ? inv : rinv;
#pragma unroll
        for (int c = j + 1; c < SB; ++c) s[c] = fmaf(-l, __shfl_sync(kFull, l, c), s[c]);
      }
      if (bad >= 0 && o + bad < b && lane == 0)
        report_error(st, KFAC_ERR_NOT_PD, J.layer, k + o + bad);
      if (lane < SB) {
#pragma unroll
        for (int c = 0; c < SB; ++c)
          if (c <= r) A[(o + r) * AP + o + c] = s[c];
        X[(o + r) * AP + o + r] = rinv;   // X_kk's diagonal
      }
    }
    __syncthreads();
    const int nr = NB - o - SB;   // rows below the sub-block
    if (nr > 0) {
      // (b) the rows below: L_below = A_below L_D^{-T}, one thread per row by
      // forward substitution, x_c = (a_c - sum_{m<c} x_m L_D[c][m]) / L_D[c][c]
      if (tid < nr) {
        const int i = o + SB + tid;
        float x[SB];
#pragma unroll
        for (int c = 0; c < SB; ++c) x[c] = A[i * AP + o + c];
#pragma unroll
        for (int c = 0; c < SB; ++c) {
          float a0 = x[c], a1 = 0.f;   // two chains
#pragma unroll
          for (int m = 0; m < c; ++m) {
            if (m & 1) a1 = fmaf(-x[m], A[(o + c) * AP + o + m], a1);
            else a0 = fmaf(-x[m], A[(o + c) * AP + o + m], a0);
          }
          x[c] = (a0 + a1) * X[(o + c) * AP + o + c];
        }
#pragma unroll
        for (int c = 0; c < SB; ++c) A[i * AP + o + c] = x[c];
      }
      __syncthreads();
      // (c) thread: column jj with row jj of L_below in registers; rows i >= jj
      const int jj = o + SB + (tid & 63);
      if (jj < NB) {
        float lj[SB];
#pragma unroll
        for (int m = 0; m < SB; ++m) lj[m] = A[jj * AP + o + m];
        for (int i = o + SB + (tid >> 6); i < NB; i += 4) {
          if (i < jj) continue;
          float acc = A[i * AP + jj];
#pragma unroll
          for (int m = 0; m < SB; ++m) acc = fmaf(-A[i * AP + o + m], lj[m], acc);
          A[i * AP + jj] = acc;
        }
      }
      __syncthreads();
    }
  }
  // X_kk = L_kk^{-1} from its diagonal by doubling over block pairs of size 1 to 32
  diag_inverse_level<1>(A, X, Y, tid);
  diag_inverse_level<2>(A, X, Y, tid);
  diag_inverse_level<4>(A, X, Y, tid);
  diag_inverse_level<8>(A, X, Y, tid);
  diag_inverse_level<SB>(A, X, Y, tid);
  diag_inverse_level<2 * SB>(A, X, Y, tid);
  if (b == NB) {   // a whole block: constant index arithmetic
#pragma unroll
    for (int u = 0; u < NB * NB / 256; ++u) {
      const int e = tid + 256 * u;
      const int r = e / NB, c = e % NB;
      const int64_t g = (int64_t)(k + r) * n + k + c;
      J.L[g] = (c <= r) ? A[r * AP + c] : 0.f;
      J.X[g] = (c <= r) ? X[r * AP + c] : 0.f;
    }
    return;
  }
#pragma unroll 4
  for (int e = tid; e < b * b; e += 256) {
    const int r = e / b, c = e % b;
    const int64_t g = (int64_t)(k + r) * n + k + c;
    J.L[g] = (c <= r) ? A[r * AP + c] : 0.f;
    J.X[g] = (c <= r) ? X[r * AP + c] : 0.f;
  }
}

// L[i, k:k+b] <- L[i, k:k+b] . X_kk^T for rows i in [k+b, n); one CTA owns a
// 64-row block and all b <= 64 columns, so the in-place update is race-free.
__global__ void __launch_bounds__(256) chol_panel_kernel(const InvJob* jobs, int k) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int n = J.n;
  if (k + NB >= n) return;  // no rows below the last diagonal block
  const int b = NB;
  const int64_t r0 = (int64_t)k + b + (int64_t)blockIdx.x * 64;
  if (r0 >= n) return;
  __shared__ float smem[PTile::kSmemFloats];
  float acc[4][4] = {};
  StridedLoader la{J.L + k, n, 1, n, b};                       // (r, t) -> L[r][k+t]
  StridedLoader lb{J.X + (int64_t)k * n + k, 1, n, b, b};      // (t, c) -> X[k+c][k+t]
  PTile::run<true, true>(la, lb, r0, 0, 0, b, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = r0 + PTile::row_of(i);
      const int c = PTile::col_of(j);
      if (r < n && c < b) J.L[r * n + k + c] = acc[i][j];
    }
}

// L[i][j] -= sum_t L[i][k+t] L[j][k+t] over the trailing lower tiles (ti >= tj,
// counted from the first trailing block), for block columns below `cend` (the
// end of the current outer panel; the tensor cores update the rest).  part: 1
// the first block column only (tj = 0: what the next diagonal block and panel
// need); 2 the others (tj >= 1), which may run alongside the next diagonal
// block and panel.
__global__ void __launch_bounds__(256) chol_trailing_kernel(const InvJob* jobs, int k, int part,
                                                            int cend) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int n = J.n;
  const int64_t base = (int64_t)k + NB;
  if (base >= n) return;
  const int nt = (int)((n - base + 63) / 64);
  const int nc = min(nt, (int)((min(cend, n) - base + 63) / 64));   // block columns to update
  if (nc <= 0) return;
  int ti, tj;
  if (part == 1) {
    if ((int)blockIdx.x >= nt) return;
    ti = blockIdx.x;
    tj = 0;
  } else {
    int t = blockIdx.x, j = 1;
    for (; j < nc; ++j) {
      if (t < nt - j) break;
      t -= nt - j;
    }
    if (j >= nc) return;
    tj = j;
    ti = j + t;
  }
  __shared__ float smem[PTile::kSmemFloats];
  float acc[4][4] = {};
  StridedLoader la{J.L + k, n, 1, n, NB};   // (i, t) -> L[i][k+t]
  StridedLoader lb{J.L + k, 1, n, NB, n};   // (t, j) -> L[j][k+t]
  PTile::run<true, true>(la, lb, base + ti * 64, base + tj * 64, 0, NB, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = base + ti * 64 + PTile::row_of(i);
      const int64_t c = base + tj * 64 + PTile::col_of(j);
      if (r < n && c < n) J.L[r * n + c] -= acc[i][j];
    }
}

// Locate the (pair, tile) of a CTA at doubling level s.  Pair p: T = [2ps, (2p+1)s),
// B = [(2p+1)s, min((2p+2)s, n)); tiles cover B rows x T cols in 64 x 64 blocks.
__device__ __forceinline__ bool level_tile(int n, int s, int t, int* T0, int* B0, int* B1,
                                           int* tr, int* tc) {
  for (int p = 0;; ++p) {
    const int t0 = 2 * p * s, b0 = t0 + s;
    if (b0 >= n) return false;
    const int b1 = min(b0 + s, n);
    const int rows = (b1 - b0 + 63) / 64, cols = s / 64;
    if (t < rows * cols) {
      *T0 = t0;
      *B0 = b0;
      *B1 = b1;
      *tr = t / cols;
      *tc = t % cols;
      return true;
    }
    t -= rows * cols;
  }
}

// Y[r][c] = sum_{t in T, t >= c} L[r][t] X[t][c]      (r in B, c in T)
__global__ void __launch_bounds__(256) tri_level_y_kernel(const InvJob* jobs, int s) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int n = J.n;
  int T0, B0, B1, tr, tc;
  if (!level_tile(n, s, blockIdx.x, &T0, &B0, &B1, &tr, &tc)) return;
  __shared__ float smem[PTile::kSmemFloats];
  float acc[4][4] = {};
  StridedLoader la{J.L, n, 1, B1, T0 + s};   // (r, t) -> L[r][t]
  StridedLoader lb{J.X, n, 1, T0 + s, T0 + s};  // (t, c) -> X[t][c]
  const int64_t m0 = B0 + tr * 64, c0 = T0 + tc * 64;
  PTile::run<true, false>(la, lb, m0, c0, c0, T0 + s, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = m0 + PTile::row_of(i), c = c0 + PTile::col_of(j);
      if (r < B1) J.Y[r * n + c] = acc[i][j];
    }
}

// X[r][c] = -sum_{t in B, t <= r} X[r][t] Y[t][c]      (r in B, c in T)
__global__ void __launch_bounds__(256) tri_level_x_kernel(const InvJob* jobs, int s) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int n = J.n;
  int T0, B0, B1, tr, tc;
  if (!level_tile(n, s, blockIdx.x, &T0, &B0, &B1, &tr, &tc)) return;
  __shared__ float smem[PTile::kSmemFloats];
  float acc[4][4] = {};
  StridedLoader la{J.X, n, 1, B1, B1};      // (r, t) -> X[r][t]
  StridedLoader lb{J.Y, n, 1, B1, T0 + s};  // (t, c) -> Y[t][c]
  const int64_t m0 = B0 + tr * 64, c0 = T0 + tc * 64;
  const int64_t k1 = m0 + 64 < (int64_t)B1 ? m0 + 64 : (int64_t)B1;
  PTile::run<true, false>(la, lb, m0, c0, B0, k1, acc, smem);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t r = m0 + PTile::row_of(i), c = c0 + PTile::col_of(j);
      if (r < B1) J.X[r * n + c] = -acc[i][j];
    }
}

// Outer-panel operand for the tensor-core trailing update: the panel's rows
// below it, P = L[cend:, K0:K0+W], already K-major (rows of L), split into TF32
// halves with pitch W.
struct PanelPack {
  const float* src;
  int64_t ld, rows;
  float* hi;
  float* lo;
};
constexpr int kMaxPanelPacks = 32;
struct PanelPackGroup {
  PanelPack job[kMaxPanelPacks];
  int count, W;
};

__global__ void __launch_bounds__(256) panel_split_kernel(const __grid_constant__ PanelPackGroup g) {
  pdl_wait();
  pdl_trigger();
  const PanelPack P = g.job[blockIdx.y];
  for (int64_t r = blockIdx.x; r < P.rows; r += gridDim.x) {
#pragma unroll 2
    for (int c = threadIdx.x; c < g.W; c += blockDim.x) {
      const float v = P.src[r * P.ld + c];
      const float hi = tc::to_tf32(v);
      P.hi[r * g.W + c] = hi;
      P.lo[r * g.W + c] = tc::to_tf32(v - hi);
    }
  }
}

// Finv -> the operand form of the K4 products (the inverses are their B
// operands): TF32 hi and bf16 correction pairs (tc::corr_pair, B form) with a
// 16-byte row pitch (np), or, for bf16 preconditioning, bf16 values in the hi
// array with a row pitch of 2 np elements.
__global__ void __launch_bounds__(256) inv_split_kernel(const InvJob* jobs, int bf16) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(J.Finv_hi);
  for (int64_t r = blockIdx.x; r < J.n; r += gridDim.x) {
    const float* src = J.Finv + r * J.n;
    if (bf16) {
      __nv_bfloat16* d = ob + r * 2 * J.np;
#pragma unroll 4
      for (int c = threadIdx.x; c < J.n; c += blockDim.x) d[c] = __float2bfloat16_rn(src[c]);
      continue;
    }
    float* dh = J.Finv_hi + r * J.np;
    uint32_t* dl = reinterpret_cast<uint32_t*>(J.Finv_lo) + r * J.np;
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) dh[c] = tc::corr_pair(src[c], true, &dl[c]);
  }
}

// Operands of the tensor-core doubling levels: blocks of L and X split into TF32
// halves, dst[r][c] (row pitch dp) = src[r][c], or src[c][r] for a transposed
// block.  One CTA moves a 64 x 64 tile through shared memory (loads and stores
// both coalesced).
struct BlockPack {
  const float* src;   // block origin, row pitch ld
  int64_t ld;
  float* hi;
  float* lo;
  int64_t dp;
  int rows, cols;     // of the destination block
  int trans;          // 1: dst[r][c] = src[c * ld + r]
};
constexpr int kMaxBlockPacks = 192;
struct BlockPackGroup {
  BlockPack job[kMaxBlockPacks];
  int tile_start[kMaxBlockPacks + 1];
  int count;
};

constexpr int kBP = 64;   // block-pack tile: 64 x 64, 16 loads in flight per thread
__global__ void __launch_bounds__(256) block_pack_kernel(const __grid_constant__ BlockPackGroup g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float t[kBP][kBP + 1];
  const int b = blockIdx.x;
  int q = 0;
  while (q + 1 < g.count && b >= g.tile_start[q + 1]) ++q;
  const BlockPack J = g.job[q];
  const int local = b - g.tile_start[q];
  const int tcols = (J.cols + kBP - 1) / kBP;
  const int tr = local / tcols, tcl = local % tcols;   // destination tile
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  float v[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int i = ty + 8 * (u >> 1), j = tx + 32 * (u & 1);
    v[u] = 0.f;
    if (!J.trans) {   // source row i of the tile = destination row i
      const int r = tr * kBP + i, c = tcl * kBP + j;
      if (r < J.rows && c < J.cols) v[u] = J.src[(int64_t)r * J.ld + c];
    } else {          // source row i of the tile = destination column i
      const int r = tr * kBP + j, c = tcl * kBP + i;
      if (r < J.rows && c < J.cols) v[u] = J.src[(int64_t)c * J.ld + r];
    }
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int i = ty + 8 * (u >> 1), j = tx + 32 * (u & 1);
    if (!J.trans) t[i][j] = v[u];
    else t[j][i] = v[u];
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int i = ty + 8 * (u >> 1), j = tx + 32 * (u & 1);
    const int r = tr * kBP + i, c = tcl * kBP + j;
    if (r >= J.rows || c >= J.cols) continue;
    const float w = t[i][j];
    const float hi = tc::to_tf32(w);
    J.hi[(int64_t)r * J.dp + c] = hi;
    J.lo[(int64_t)r * J.dp + c] = tc::to_tf32(w - hi);
  }
}

int level_tiles_host(int n, int s) {
  int total = 0;
  for (int p = 0;; ++p) {
    const int b0 = (2 * p + 1) * s;
    if (b0 >= n) break;
    const int b1 = std::min(b0 + s, n);
    total += ((b1 - b0 + 63) / 64) * (s / 64);
  }
  return total;
}

}  // namespace

size_t inv_y_floats(int n) { return (size_t)n * n; }

// One doubling level on the tensor cores, for every factor with pairs at this
// level (pair (T, B): T = [t0, t0 + s), B = [b0, b1), b0 = t0 + s):
//   Y^T  = (L_BT X_TT)^T         product 1: A = L_BT, B = X_TT^T, K = s; stored as
//                                TF32 halves (the next product's operand)
//   X_BT = -(Y^T X_BB^T)^T        product 2: A = Y^T, B = X_BB, K = |B|; stored as
//                                fp32 straight into X (transposed store, alpha = -1)
// The operand blocks (L_BT, X_TT^T, X_BB as TF32 halves) are packed first.
// Scratch per factor: L_BT and Y^T halves in its Y buffer (n^2 floats), X_TT^T
// and X_BB halves in its inverse halves (n x np each, written only after the
// levels).  Returns KFAC_ERR_WORKSPACE, before any launch, when a factor's
// blocks do not fit: the caller then runs the level on the CUDA cores.
kfac_status launch_tri_level_tc(kfac_ctx* h, int j0, int nj, int s, cudaStream_t st) {
  struct PairOps {
    BlockPack lbt, xtt, xbb;
    TcProblem p1, p2;
  };
  std::vector<PairOps> ops;
  auto al = [](size_t f) { return (f + 31) / 32 * 32; };   // 128-byte aligned sub-buffers
  for (int i = j0; i < j0 + nj; ++i) {
    const InvJob& J = h->invjobs_host[i];
    const int n = J.n;
    size_t yoff = 0, foff = 0;
    for (int p = 0;; ++p) {
      const int t0 = 2 * p * s, b0 = t0 + s;
      if (b0 >= n) break;
      const int b1 = std::min(b0 + s, n), mb = b1 - b0;
      const int64_t mbp = tc_pitch(mb, false);
      float* lbt_hi = J.Y + yoff;
      float* lbt_lo = lbt_hi + al((size_t)mb * s);
      float* yt_hi = lbt_lo + al((size_t)mb * s);
      float* yt_lo = yt_hi + al((size_t)s * mbp);
      yoff += 2 * al((size_t)mb * s) + 2 * al((size_t)s * mbp);
      float* xtt_hi = J.Finv_hi + foff;
      float* xtt_lo = J.Finv_lo + foff;
      float* xbb_hi = xtt_hi + al((size_t)s * s);
      float* xbb_lo = xtt_lo + al((size_t)s * s);
      foff += al((size_t)s * s) + al((size_t)mb * mbp);
      if (yoff > inv_y_floats(n) || foff > (size_t)n * J.np) return KFAC_ERR_WORKSPACE;
      PairOps o{};
      o.lbt = BlockPack{J.L + (int64_t)b0 * n + t0, n, lbt_hi, lbt_lo, s, mb, s, 0};
      o.xtt = BlockPack{J.X + (int64_t)t0 * n + t0, n, xtt_hi, xtt_lo, s, s, s, 1};
      o.xbb = BlockPack{J.X + (int64_t)b0 * n + b0, n, xbb_hi, xbb_lo, mbp, mb, mb, 0};
      o.p1.A = TcOperand{lbt_hi, lbt_lo, mb, s};
      o.p1.B = TcOperand{xtt_hi, xtt_lo, s, s};
      o.p1.M = mb;
      o.p1.N = s;
      o.p1.K = s;
      o.p1.e.out_hi = yt_hi;
      o.p1.e.out_lo = yt_lo;
      o.p1.e.ldo = mbp;
      o.p1.layer = J.layer;
      o.p1.kmode = 1;   // X_TT lower: column c sums over t >= c
      o.p2.A = TcOperand{yt_hi, yt_lo, s, mbp};
      o.p2.B = TcOperand{xbb_hi, xbb_lo, mb, mbp};
      o.p2.M = s;
      o.p2.N = mb;
      o.p2.K = mb;
      o.p2.e.out_hi = J.X + (int64_t)b0 * n + t0;
      o.p2.e.out_lo = nullptr;
      o.p2.e.ldo = n;
      o.p2.e.alpha = -1.f;
      o.p2.layer = J.layer;
      o.p2.kmode = 2;   // X_BB lower: column r sums over t <= r
      ops.push_back(o);
    }
  }
  if (ops.empty()) return KFAC_OK;
  // packs, in launches of up to kMaxBlockPacks blocks
  std::unique_ptr<BlockPackGroup> g(new BlockPackGroup());
  std::memset(g.get(), 0, sizeof(BlockPackGroup));
  int tiles = 0;
  auto flush = [&]() -> kfac_status {
    if (g->count == 0) return KFAC_OK;
    g->tile_start[g->count] = tiles;
    launch_pdl(block_pack_kernel, dim3((unsigned)tiles), dim3(256), 0, st, *g);
    count_launch();
    std::memset(g.get(), 0, sizeof(BlockPackGroup));
    tiles = 0;
    return check_launch();
  };
  auto add = [&](const BlockPack& b) -> kfac_status {
    if (g->count == kMaxBlockPacks)
      if (kfac_status e = flush()) return e;
    g->job[g->count] = b;
    g->tile_start[g->count] = tiles;
    tiles += (int)(cdiv(b.rows, kBP) * cdiv(b.cols, kBP));
    ++g->count;
    return KFAC_OK;
  };
  std::vector<TcProblem> p1, p2;
  for (const PairOps& o : ops) {
    for (const BlockPack* b : {&o.lbt, &o.xtt, &o.xbb})
      if (kfac_status e = add(*b)) return e;
    p1.push_back(o.p1);
    p2.push_back(o.p2);
  }
  if (kfac_status e = flush()) return e;
  if (kfac_status e = launch_gemm_tc_grouped(h, false, TC_EPI_SPLIT, p1.data(), (int)p1.size(), st))
    return e;
  return launch_gemm_tc_grouped(h, false, TC_EPI_SPLIT, p2.data(), (int)p2.size(), st);
}

// L22 <- L22 - P P^T for every factor whose size reaches past the outer panel
// [K0, K0 + W): P = L[K0 + W :, K0 : K0 + W] split into TF32 halves, then one
// grouped 3xTF32 SYRK (upper tiles + mirror; the trailing block is kept
// symmetric, so either triangle holds the old values).  Groups are cut where
// the pack scratch is full.
kfac_status launch_outer_update(kfac_ctx* h, int j0, int nj, int K0, int W, cudaStream_t st) {
  const int cend = K0 + W;
  PanelPackGroup pg;
  std::memset(&pg, 0, sizeof(pg));
  pg.W = W;
  std::vector<TcProblem> pr;
  size_t used = 0;
  int64_t max_elems = 0;
  auto flush = [&]() -> kfac_status {
    if (pr.empty()) return KFAC_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(cdiv(max_elems, 256), 4 * num_sms());
    launch_pdl(panel_split_kernel, dim3(dim3(blocks, pg.count)), dim3(256), 0, st, pg);
    count_launch();
    kfac_status e = check_launch();
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, false, TC_EPI_SYRK, pr.data(), (int)pr.size(), st);
    pr.clear();
    pg.count = 0;
    used = 0;
    max_elems = 0;
    return e;
  };
  for (int i = j0; i < j0 + nj; ++i) {
    const InvJob& J = h->invjobs_host[i];
    if (J.n <= cend) continue;
    const int64_t m = J.n - cend;
    const size_t raw = (size_t)m * W * 8, bytes = align_up(raw);
    if (raw > h->tcpack_bytes) return KFAC_ERR_WORKSPACE;
    if (used + raw > h->tcpack_bytes || pg.count == kMaxPanelPacks)
      if (kfac_status e = flush()) return e;
    float* hi = reinterpret_cast<float*>(h->ws + h->off_tcpack + used);
    float* lo = hi + (size_t)m * W;
    used += bytes;
    PanelPack& pp = pg.job[pg.count++];
    pp.src = J.L + (int64_t)cend * J.n + K0;
    pp.ld = J.n;
    pp.rows = m;
    pp.hi = hi;
    pp.lo = lo;
    max_elems = std::max<int64_t>(max_elems, m * W);
    TcProblem t{};
    t.A = TcOperand{hi, lo, m, W};
    t.B = t.A;
    t.same_ab = true;
    t.upper = true;
    t.M = t.N = m;
    t.K = W;
    t.e.alpha = -1.f;
    t.e.beta = 1.f;
    t.e.C = J.L + (int64_t)cend * J.n + cend;
    t.e.ldc = J.n;
    t.layer = J.layer;
    pr.push_back(t);
  }
  return flush();
}

// Inside an outer panel: L[e:, e:c] <- L[e:, e:c] - P Q^T for every factor whose
// size reaches past e = H0 + MW, with P = L[e:, H0:e] (MW columns, split into
// TF32 halves) and Q = its rows [e, c) (c the end of the outer panel): one
// grouped 3xTF32 product with the transposed fp32 store accumulating into L
// (C^T = Q P^T, alpha -1, beta 1).  Q's rows are the first of P's, so one pack
// serves both operands.  The square [e, c)^2 gets both triangles, which keeps
// it symmetric for the steps that factor it.
kfac_status launch_mid_update(kfac_ctx* h, int j0, int nj, int H0, int MW, int c,
                              cudaStream_t st) {
  const int e0 = H0 + MW;
  PanelPackGroup pg;
  std::memset(&pg, 0, sizeof(pg));
  pg.W = MW;
  std::vector<TcProblem> pr;
  size_t used = 0;
  int64_t max_rows = 0;
  auto flush = [&]() -> kfac_status {
    if (pr.empty()) return KFAC_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(max_rows, 4 * num_sms());
    launch_pdl(panel_split_kernel, dim3(dim3(blocks, pg.count)), dim3(256), 0, st, pg);
    count_launch();
    kfac_status e = check_launch();
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, false, TC_EPI_SPLIT, pr.data(), (int)pr.size(), st);
    pr.clear();
    pg.count = 0;
    used = 0;
    max_rows = 0;
    return e;
  };
  for (int i = j0; i < j0 + nj; ++i) {
    const InvJob& J = h->invjobs_host[i];
    if (J.n <= e0) continue;
    const int64_t m = J.n - e0;
    const size_t raw = (size_t)m * MW * 8, bytes = align_up(raw);
    if (raw > h->tcpack_bytes) return KFAC_ERR_WORKSPACE;
    if (used + raw > h->tcpack_bytes || pg.count == kMaxPanelPacks)
      if (kfac_status e = flush()) return e;
    float* hi = reinterpret_cast<float*>(h->ws + h->off_tcpack + used);
    float* lo = hi + (size_t)m * MW;
    used += bytes;
    PanelPack& pp = pg.job[pg.count++];
    pp.src = J.L + (int64_t)e0 * J.n + H0;
    pp.ld = J.n;
    pp.rows = m;
    pp.hi = hi;
    pp.lo = lo;
    max_rows = std::max<int64_t>(max_rows, m);
    TcProblem t{};
    t.A = TcOperand{hi, lo, std::min<int64_t>(c, J.n) - e0, MW};   // Q: rows [e0, c)
    t.B = TcOperand{hi, lo, m, MW};                                   // P: rows [e0, n)
    t.M = t.A.rows;
    t.N = m;
    t.K = MW;
    t.e.alpha = -1.f;
    t.e.beta = 1.f;
    t.e.out_hi = J.L + (int64_t)e0 * J.n + e0;   // C^T[c][r] = L[e0 + c][e0 + r]
    t.e.ldo = J.n;
    t.layer = J.layer;
    pr.push_back(t);
  }
  return flush();
}

kfac_status launch_ikfac_seed(const InvJob* jobs, int nj, int nmax, bool bf16, cudaStream_t st);

kfac_status launch_invert(kfac_ctx* h, int layer, int which, cudaStream_t st) {
  // job range: the table section of the wanted factors (both, A only, G only),
  // whole or the entries of one layer (contiguous: a section is in layer order)
  const InvJob* d_all = h->at<InvJob>(h->off_invjobs);
  const SyrkJob* d_syrk = h->at<SyrkJob>(h->off_invjobs + align_up(sizeof(InvJob) * h->n_invjobs));
  const int sec = which == (KFAC_FACTOR_A | KFAC_FACTOR_G) ? 0 : which == KFAC_FACTOR_A ? 1 : 2;
  int j0 = h->tab_start[sec], nj = h->tab_count[sec];
  if (layer >= 0) {
    int first = -1, cnt = 0;
    for (int i = j0; i < j0 + nj; ++i)
      if (h->invjobs_host[i].layer == layer) {
        if (first < 0) first = i;
        ++cnt;
      }
    j0 = first;
    nj = cnt;
  }
  if (nj == 0) return KFAC_OK;   // nothing of that kind to refresh (a tied A)
  int nmax = 0;
  for (int i = j0; i < j0 + nj; ++i) nmax = std::max(nmax, h->invjobs_host[i].n);
  const InvJob* jobs = d_all + j0;
  const float sg = (float)std::sqrt(h->hp.damping);

  launch_pdl(inv_prep_kernel, dim3(dim3((unsigned)std::min<int64_t>(cdiv((int64_t)nmax * nmax, 256), 1024), nj)), dim3(256), 0, st, jobs, sg);
  count_launch();
  if (kfac_status e = check_launch()) return e;

  // Cholesky in outer panels of kOuterW columns (the whole matrix when every
  // factor is at most kOuterMaxN): inside a panel, 64-column steps with one
  // block of lookahead -- after the panel of step k, the trailing update of the
  // next block column runs on the caller's stream (the next diagonal block
  // needs it), the panel's other columns on the side stream, concurrently with
  // the next diagonal block and panel (events: the side stream waits for each
  // panel; the next block column's update waits for the previous side work,
  // which also writes that column).  After each outer panel the tensor cores
  // update the whole trailing block with it: L22 <- L22 - P P^T, K = kOuterW.
  bool rest_pending = false;
  auto sync_err = [](cudaError_t e) { return e == cudaSuccess ? KFAC_OK : KFAC_ERR_CUDA; };
  auto join_side = [&]() -> kfac_status {
    if (!rest_pending) return KFAC_OK;
    rest_pending = false;
    return sync_err(cudaStreamWaitEvent(st, h->ev_rest, 0));
  };
  const int W = nmax > kOuterMaxN ? kOuterW : (int)cdiv(nmax, NB) * NB;
  const int MW = W == kOuterW ? kMidW : W;   // inner steps update their half panel only
  for (int K0 = 0; K0 < nmax; K0 += W) {
   for (int H0 = K0; H0 < std::min(K0 + W, nmax); H0 += MW) {
    const int cend = H0 + MW;   // the inner steps' trailing updates stop here
    for (int k = H0; k < std::min(cend, nmax); k += NB) {
      launch_pdl(chol_diag_kernel, dim3(nj), dim3(256), 0, st, jobs, k, h->status());
      count_launch();
      const int rest = nmax - k - NB;
      if (rest > 0) {
        const int rb = (int)cdiv(rest, 64);
        launch_pdl(chol_panel_kernel, dim3(dim3(rb, nj)), dim3(256), 0, st, jobs, k);
        count_launch();
        const int nc = (int)std::min<int64_t>(rb, cdiv(std::min(cend, nmax) - (k + NB), 64));
        if (nc > 1) {
          if (kfac_status e = sync_err(cudaEventRecord(h->ev_panel, st))) return e;
          if (kfac_status e = sync_err(cudaStreamWaitEvent(h->side_stream, h->ev_panel, 0))) return e;
        }
        if (nc >= 1) {
          if (kfac_status e = join_side()) return e;
          launch_pdl(chol_trailing_kernel, dim3(dim3(rb, nj)), dim3(256), 0, st, jobs, k, 1, cend);
          count_launch();
        }
        if (nc > 1) {
          int64_t tiles = 0;
          for (int j = 1; j < nc; ++j) tiles += rb - j;
          launch_pdl(chol_trailing_kernel, dim3(dim3((unsigned)tiles, nj)), dim3(256), 0, h->side_stream, jobs, k, 2, cend);
          count_launch();
          if (kfac_status e = sync_err(cudaEventRecord(h->ev_rest, h->side_stream))) return e;
          rest_pending = true;
        }
      }
      if (kfac_status e = check_launch()) return e;
    }
    if (cend < std::min(K0 + W, nmax)) {   // the second half of the outer panel
      if (kfac_status e = join_side()) return e;
      if (kfac_status e = launch_mid_update(h, j0, nj, H0, MW, K0 + W, st)) return e;
    }
   }
    if (K0 + W < nmax) {
      if (kfac_status e = join_side()) return e;
      if (kfac_status e = launch_outer_update(h, j0, nj, K0, W, st)) return e;
    }
  }
  if (kfac_status e = join_side()) return e;
  for (int s = NB; s < nmax; s *= 2) {
    // the wide levels on the tensor cores, when they carry a few waves of work:
    // at least about four 128 x 128 x 512 tiles per SM over all factors' pairs
    // (smaller levels run faster as the CUDA-core tiles below)
    double level_fma = 0;
    for (int i = j0; i < j0 + nj; ++i) {
      const int n = h->invjobs_host[i].n;
      for (int b0 = s; b0 < n; b0 += 2 * s) level_fma += 2.0 * (double)s * s * std::min(s, n - b0);
    }
    if (s >= kTcLevelMin && level_fma >= 4.0 * num_sms() * 128 * 128 * 512) {
      kfac_status e = launch_tri_level_tc(h, j0, nj, s, st);
      if (e == KFAC_OK) continue;
      if (e != KFAC_ERR_WORKSPACE) return e;
    }
    const int tiles = level_tiles_host(nmax, s);
    int tmax = tiles;
    for (int i = j0; i < j0 + nj; ++i) tmax = std::max(tmax, level_tiles_host(h->invjobs_host[i].n, s));
    launch_pdl(tri_level_y_kernel, dim3(dim3(tmax, nj)), dim3(256), 0, st, jobs, s);
    launch_pdl(tri_level_x_kernel, dim3(dim3(tmax, nj)), dim3(256), 0, st, jobs, s);
    count_launch(2);
    if (kfac_status e = check_launch()) return e;
  }
  // F_d^{-1} = X^T X: small factors in one grouped CUDA-core launch, large ones on the
  // tensor cores (pack X^T into TF32 halves, 3xTF32 SYRK)
  int nt_small = 0;
  for (int i = j0; i < j0 + nj; ++i)
    if (h->invjobs_host[i].n < kTcInverseMinN)
      nt_small = std::max(nt_small, (int)cdiv(h->invjobs_host[i].n, SyrkTile::BM));
  if (nt_small > 0)
    if (kfac_status e = launch_syrk_simt_grouped(d_syrk + j0, nj, nt_small * (nt_small + 1) / 2, st))
      return e;
  std::vector<SyrkSpec> big;
  for (int i = j0; i < j0 + nj; ++i) {
    const InvJob& J = h->invjobs_host[i];
    if (J.n < kTcInverseMinN) continue;
    big.push_back(SyrkSpec{J.X, J.n, J.n, J.n, J.n, J.layer, 1.f, 0.f, J.Finv, 1});   // X lower
  }
  if (!big.empty())
    if (kfac_status e = launch_syrk_tc_batched(h, big.data(), (int)big.size(), st)) return e;
  launch_pdl(inv_split_kernel, dim3(dim3((unsigned)std::min<int64_t>(cdiv((int64_t)nmax * nmax, 256), 1024), nj)), dim3(256), 0, st, jobs,
             (int)(h->hp.math == KFAC_MATH_BF16));
  count_launch();
  if (kfac_status e = check_launch()) return e;
  // inverse-free update: K = X^T (so K K^T = X^T X = F_d^{-1}), and K^T = X
  if (h->hp.ikfac) return launch_ikfac_seed(jobs, nj, nmax, h->hp.ikfac == KFAC_IKFAC_BF16, st);
  return KFAC_OK;
}

// ---------------------------------------------------------------------------
// Inverse-free update ("Structured Inverse-Free Natural Gradient" page,
// abstract: an inverse-free K-FAC update by subtraction in the matrix-logarithm
// space).  Per factor, K (K K^T standing for F_d^{-1}) takes the step
//   K <- K (I - (beta/2)(K^T F_d K - I))
// as tensor-core products with the transposed-store epilogue (C = A B^T on
// K-major TF32-half operands, C^T stored as halves):
//   S1 <- F_d                    (damped, split)
//   S2 <- (F_d K)^T              A = S1, B = K^T
//   S1 <- (K^T F_d K)^T          A = K^T, B = S2
//   S1 <- (1 + beta/2) I - (beta/2) S1          (= M^T)
//   K^T <- (K M)^T               A = K, B = S1
//   K <- (K^T)^T                 (transpose of the halves)
//   F_d^{-1} <- K K^T            SYRK, A = B = K; then its halves for K4.
// Every array is n x np (np = n rounded up to 4, the TMA row pitch).

namespace {

constexpr int kTT = 32;   // transpose tile

// K^T = X (lower, pitch n) and K = X^T, as TF32 halves.
__global__ void __launch_bounds__(256) ik_seed_kernel(const InvJob* jobs) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int tn = (J.n + kTT - 1) / kTT;
  if ((int)blockIdx.x >= tn * tn) return;
  const int r0 = (blockIdx.x / tn) * kTT, c0 = (blockIdx.x % tn) * kTT;
  __shared__ float t[kTT][kTT + 1];
  const int tx = threadIdx.x % kTT, ty = threadIdx.x / kTT;   // 32 x 8
  for (int rr = ty; rr < kTT; rr += 8) {
    const int r = r0 + rr, c = c0 + tx;
    float v = 0.f;
    if (r < J.n && c < J.n) {
      v = J.X[(int64_t)r * J.n + c];
      const float hi = tc::to_tf32(v);
      J.Kt_hi[(int64_t)r * J.np + c] = hi;
      J.Kt_lo[(int64_t)r * J.np + c] = tc::to_tf32(v - hi);
    }
    t[rr][tx] = v;
  }
  __syncthreads();
  for (int cc = ty; cc < kTT; cc += 8) {   // K[c][r] = X[r][c]
    const int c = c0 + cc, r = r0 + tx;
    if (r < J.n && c < J.n) {
      const float v = t[tx][cc];
      const float hi = tc::to_tf32(v);
      J.K_hi[(int64_t)c * J.np + r] = hi;
      J.K_lo[(int64_t)c * J.np + r] = tc::to_tf32(v - hi);
    }
  }
}

// S1 <- split(F + sqrt(gamma) I)  (F: running factor, pitch n)
__global__ void __launch_bounds__(256) ik_damped_split_kernel(const InvJob* jobs, float sqrt_gamma) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  for (int64_t r = blockIdx.x; r < J.n; r += gridDim.x)
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) {
      const float v = J.F[r * J.n + c] + (r == c ? sqrt_gamma : 0.f);
      const float hi = tc::to_tf32(v);
      J.S1_hi[r * J.np + c] = hi;
      J.S1_lo[r * J.np + c] = tc::to_tf32(v - hi);
    }
}

// S1 <- split(c1 I - c2 S1)
__global__ void __launch_bounds__(256) ik_affine_kernel(const InvJob* jobs, float c1, float c2) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  for (int64_t r = blockIdx.x; r < J.n; r += gridDim.x)
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) {
      const int64_t x = r * J.np + c;
      const float v = fmaf(-c2, J.S1_hi[x] + J.S1_lo[x], r == c ? c1 : 0.f);
      const float hi = tc::to_tf32(v);
      J.S1_hi[x] = hi;
      J.S1_lo[x] = tc::to_tf32(v - hi);
    }
}

// K <- (K^T)^T, both halves, through 32 x 33 shared tiles
__global__ void __launch_bounds__(256) ik_transpose_kernel(const InvJob* jobs) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int tn = (J.n + kTT - 1) / kTT;
  if ((int)blockIdx.x >= tn * tn) return;
  const int r0 = (blockIdx.x / tn) * kTT, c0 = (blockIdx.x % tn) * kTT;
  __shared__ float th[kTT][kTT + 1], tl[kTT][kTT + 1];
  const int tx = threadIdx.x % kTT, ty = threadIdx.x / kTT;
  for (int rr = ty; rr < kTT; rr += 8) {
    const int r = r0 + rr, c = c0 + tx;
    const bool in = r < J.n && c < J.n;
    th[rr][tx] = in ? J.Kt_hi[(int64_t)r * J.np + c] : 0.f;
    tl[rr][tx] = in ? J.Kt_lo[(int64_t)r * J.np + c] : 0.f;
  }
  __syncthreads();
  for (int cc = ty; cc < kTT; cc += 8) {
    const int c = c0 + cc, r = r0 + tx;
    if (r < J.n && c < J.n) {
      J.K_hi[(int64_t)c * J.np + r] = th[tx][cc];
      J.K_lo[(int64_t)c * J.np + r] = tl[tx][cc];
    }
  }
}

// ---- bf16 products (handles created with ikfac = KFAC_IKFAC_BF16).  The step
// is the same; its three products run on bf16 tensor cores (fp32 accumulate)
// and the correction is added to an fp32 master of K^T:
//   FF <- [hi | lo]  of F_d in bf16 (hi = bf16(F_d), lo = bf16(F_d - hi))
//   Gb <- (F_d K)^T  = ([hi lo] [K; K])^T            (bf16; reduction length 2n)
//   G  <- (K^T F_d K)^T                               (fp32)
//   Wb <- -(beta/2) (G - I)                            (bf16)
//   D  <- (K Wb^T)^T = (K (-(beta/2) E))^T             (fp32)
//   K^T <- K^T + D (fp32 master); its bf16 copies; F_d^{-1} <- K K^T (bf16 SYRK)
// Rounding F_d to bf16 in one piece would move the iteration's fixed point by
// about 2^-8 cond(F_d)^(1/2) relative; its hi/lo pair keeps 16 mantissa bits.
// bf16 arrays share the fp32 arrays' storage with a row pitch of 2 np elements:
//   FF, Wb in S1_hi;  [K^T | K^T] in K_lo;  Gb in S2_hi;  K in K_hi;
//   G in S1_lo, D in S2_lo (fp32, pitch np);  the master K^T in Kt_hi.
__device__ __forceinline__ __nv_bfloat16* bf16_at(float* base) {
  return reinterpret_cast<__nv_bfloat16*>(base);
}

// from_x = 1: from X = L^{-1} (fp32, pitch n) after a Cholesky refresh: the master
// K^T = X, and its bf16 copies [K^T | K^T] and K.  from_x = 0: after a step: the
// master gains D, then the same copies.
__global__ void __launch_bounds__(256) ikb_set_kernel(const InvJob* jobs, int from_x) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int tn = (J.n + kTT - 1) / kTT;
  if ((int)blockIdx.x >= tn * tn) return;
  const int r0 = (blockIdx.x / tn) * kTT, c0 = (blockIdx.x % tn) * kTT;
  const int64_t pb = 2 * (int64_t)J.np;
  __shared__ float t[kTT][kTT + 1];
  const int tx = threadIdx.x % kTT, ty = threadIdx.x / kTT;   // 32 x 8
  __nv_bfloat16* kk = bf16_at(J.K_lo);
  __nv_bfloat16* kb = bf16_at(J.K_hi);
  for (int rr = ty; rr < kTT; rr += 8) {
    const int r = r0 + rr, c = c0 + tx;
    float v = 0.f;
    if (r < J.n && c < J.n) {
      const int64_t x = (int64_t)r * J.np + c;
      if (from_x) {
        v = J.X[(int64_t)r * J.n + c];
      } else {
        v = J.Kt_hi[x] + J.S2_lo[x];
      }
      J.Kt_hi[x] = v;
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      kk[(int64_t)r * pb + c] = b;
      kk[(int64_t)r * pb + J.n + c] = b;
    }
    t[rr][tx] = v;
  }
  __syncthreads();
  for (int cc = ty; cc < kTT; cc += 8) {   // K[c][r] = K^T[r][c]
    const int c = c0 + cc, r = r0 + tx;
    if (r < J.n && c < J.n) kb[(int64_t)c * pb + r] = __float2bfloat16_rn(t[tx][cc]);
  }
}

// FF <- [bf16(F_d) | bf16(F_d - bf16(F_d))]
__global__ void __launch_bounds__(256) ikb_damped_kernel(const InvJob* jobs, float sqrt_gamma) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int64_t pb = 2 * (int64_t)J.np;
  __nv_bfloat16* ff = bf16_at(J.S1_hi);
  for (int64_t r = blockIdx.x; r < J.n; r += gridDim.x)
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) {
      const float v = J.F[r * J.n + c] + (r == c ? sqrt_gamma : 0.f);
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      ff[r * pb + c] = hi;
      ff[r * pb + J.n + c] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

// Wb <- bf16(-(beta/2) (G - I)),  G fp32 in S1_lo
__global__ void __launch_bounds__(256) ikb_w_kernel(const InvJob* jobs, float half_beta) {
  pdl_wait();
  pdl_trigger();
  const InvJob J = jobs[blockIdx.y];
  const int64_t pb = 2 * (int64_t)J.np;
  __nv_bfloat16* w = bf16_at(J.S1_hi);
  for (int64_t r = blockIdx.x; r < J.n; r += gridDim.x)
#pragma unroll 4
    for (int c = threadIdx.x; c < J.n; c += blockDim.x) {
      const float g = J.S1_lo[r * J.np + c] - (r == c ? 1.f : 0.f);
      w[r * pb + c] = __float2bfloat16_rn(-half_beta * g);
    }
}

unsigned elem_blocks(int nmax) {
  return (unsigned)std::min<int64_t>(cdiv((int64_t)nmax * nmax, 256), 1024);
}
unsigned tile_blocks(int nmax) {
  const int64_t tn = cdiv(nmax, kTT);
  return (unsigned)(tn * tn);
}

}  // namespace

kfac_status launch_ikfac_seed(const InvJob* jobs, int nj, int nmax, bool bf16, cudaStream_t st) {
  if (bf16)
    launch_pdl(ikb_set_kernel, dim3(tile_blocks(nmax), nj), dim3(256), 0, st, jobs, 1);
  else
    launch_pdl(ik_seed_kernel, dim3(tile_blocks(nmax), nj), dim3(256), 0, st, jobs);
  count_launch();
  return check_launch();
}

// One inverse-free step with bf16 products (see ikb_set_kernel above).
kfac_status launch_ikfac_update_bf16(kfac_ctx* h, const InvJob* jobs, int j0, int nj, int nmax,
                                     float beta, cudaStream_t st) {
  launch_pdl(ikb_damped_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs,
             (float)std::sqrt(h->hp.damping));
  count_launch();
  if (kfac_status e = check_launch()) return e;
  std::vector<TcProblem> pr;
  auto bfp = [](float* p) { return static_cast<const void*>(p); };
  for (int which = 0; which < 3; ++which) {
    pr.clear();
    for (int i = j0; i < j0 + nj; ++i) {
      const InvJob& J = h->invjobs_host[i];
      const int64_t pb = 2 * (int64_t)J.np;
      TcProblem q{};
      q.M = q.N = J.n;
      q.layer = J.layer;
      q.e.alpha = 1.f;
      if (which == 0) {          // Gb <- (F_d K)^T: [hi lo] . [K; K], bf16 out
        q.A = TcOperand{bfp(J.S1_hi), nullptr, J.n, pb};
        q.B = TcOperand{bfp(J.K_lo), nullptr, J.n, pb};
        q.K = 2 * (int64_t)J.n;
        q.e.out_hi = J.S2_hi;
        q.e.out_bf16 = 1;
        q.e.ldo = pb;
      } else if (which == 1) {   // G <- (K^T F_d K)^T, fp32 out
        q.A = TcOperand{bfp(J.K_lo), nullptr, J.n, pb};
        q.B = TcOperand{bfp(J.S2_hi), nullptr, J.n, pb};
        q.K = J.n;
        q.e.out_hi = J.S1_lo;
        q.e.ldo = J.np;
      } else {                   // D <- (K Wb^T)^T, fp32 out
        q.A = TcOperand{bfp(J.K_hi), nullptr, J.n, pb};
        q.B = TcOperand{bfp(J.S1_hi), nullptr, J.n, pb};
        q.K = J.n;
        q.e.out_hi = J.S2_lo;
        q.e.ldo = J.np;
      }
      pr.push_back(q);
    }
    if (kfac_status e = launch_gemm_tc_grouped(h, true, TC_EPI_SPLIT, pr.data(), (int)pr.size(), st))
      return e;
    if (which == 1) {
      launch_pdl(ikb_w_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs, 0.5f * beta);
      count_launch();
      if (kfac_status e = check_launch()) return e;
    }
  }
  launch_pdl(ikb_set_kernel, dim3(tile_blocks(nmax), nj), dim3(256), 0, st, jobs, 0);
  count_launch();
  if (kfac_status e = check_launch()) return e;
  pr.clear();
  for (int i = j0; i < j0 + nj; ++i) {   // F_d^{-1} <- K K^T (bf16 SYRK, fp32 result)
    const InvJob& J = h->invjobs_host[i];
    TcProblem q{};
    q.M = q.N = q.K = J.n;
    q.layer = J.layer;
    q.A = TcOperand{bfp(J.K_hi), nullptr, J.n, 2 * (int64_t)J.np};
    q.B = q.A;
    q.same_ab = true;
    q.upper = true;
    q.e.alpha = 1.f;
    q.e.beta = 0.f;
    q.e.C = J.Finv;
    q.e.ldc = J.n;
    pr.push_back(q);
  }
  if (kfac_status e = launch_gemm_tc_grouped(h, true, TC_EPI_SYRK, pr.data(), (int)pr.size(), st))
    return e;
  launch_pdl(inv_split_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs,
             (int)(h->hp.math == KFAC_MATH_BF16));
  count_launch();
  return check_launch();
}

kfac_status launch_ikfac_update(kfac_ctx* h, int layer, float beta, cudaStream_t st) {
  // the factors: section 0 of the job table (A and G of each layer; no tied A)
  int j0 = h->tab_start[0], nj = h->tab_count[0];
  if (layer >= 0) {
    int first = -1, cnt = 0;
    for (int i = j0; i < j0 + nj; ++i)
      if (h->invjobs_host[i].layer == layer) {
        if (first < 0) first = i;
        ++cnt;
      }
    j0 = first;
    nj = cnt;
  }
  if (nj <= 0) return KFAC_OK;
  const InvJob* jobs = h->at<InvJob>(h->off_invjobs) + j0;
  int nmax = 0;
  for (int i = j0; i < j0 + nj; ++i) nmax = std::max(nmax, h->invjobs_host[i].n);
  if (h->hp.ikfac == KFAC_IKFAC_BF16)
    return launch_ikfac_update_bf16(h, jobs, j0, nj, nmax, beta, st);
  launch_pdl(ik_damped_split_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs,
             (float)std::sqrt(h->hp.damping));
  count_launch();
  if (kfac_status e = check_launch()) return e;
  // one grouped launch per product, over every factor
  auto products = [&](int which, std::vector<TcProblem>* out) {
    out->clear();
    for (int i = j0; i < j0 + nj; ++i) {
      const InvJob& J = h->invjobs_host[i];
      TcProblem q{};
      q.M = q.N = q.K = J.n;
      q.layer = J.layer;
      if (which == 3) {              // F_d^{-1} <- K K^T
        q.A = TcOperand{J.K_hi, J.K_lo, J.n, J.np};
        q.B = q.A;
        q.same_ab = true;
        q.upper = true;
        q.e.alpha = 1.f;
        q.e.beta = 0.f;
        q.e.C = J.Finv;
        q.e.ldc = J.n;
      } else {
        const float* a_hi = which == 0 ? J.S1_hi : which == 1 ? J.Kt_hi : J.K_hi;
        const float* a_lo = which == 0 ? J.S1_lo : which == 1 ? J.Kt_lo : J.K_lo;
        const float* b_hi = which == 0 ? J.Kt_hi : which == 1 ? J.S2_hi : J.S1_hi;
        const float* b_lo = which == 0 ? J.Kt_lo : which == 1 ? J.S2_lo : J.S1_lo;
        q.A = TcOperand{a_hi, a_lo, J.n, J.np};
        q.B = TcOperand{b_hi, b_lo, J.n, J.np};
        q.e.out_hi = which == 0 ? J.S2_hi : which == 1 ? J.S1_hi : J.Kt_hi;
        q.e.out_lo = which == 0 ? J.S2_lo : which == 1 ? J.S1_lo : J.Kt_lo;
        q.e.ldo = J.np;
      }
      out->push_back(q);
    }
  };
  std::vector<TcProblem> pr;
  for (int which = 0; which < 3; ++which) {
    products(which, &pr);
    if (kfac_status e = launch_gemm_tc_grouped(h, false, TC_EPI_SPLIT, pr.data(),
                                               (int)pr.size(), st))
      return e;
    if (which == 1) {   // S1 = (K^T F_d K)^T -> M^T = (1 + beta/2) I - (beta/2) S1
      launch_pdl(ik_affine_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs,
                 1.f + 0.5f * beta, 0.5f * beta);
      count_launch();
      if (kfac_status e = check_launch()) return e;
    }
  }
  launch_pdl(ik_transpose_kernel, dim3(tile_blocks(nmax), nj), dim3(256), 0, st, jobs);
  count_launch();
  if (kfac_status e = check_launch()) return e;
  products(3, &pr);
  if (kfac_status e = launch_gemm_tc_grouped(h, false, TC_EPI_SYRK, pr.data(), (int)pr.size(), st))
    return e;
  launch_pdl(inv_split_kernel, dim3(elem_blocks(nmax), nj), dim3(256), 0, st, jobs,
             (int)(h->hp.math == KFAC_MATH_BF16));
  count_launch();
  return check_launch();
}

}  // namespace kfac
