// FP32 CUDA-core tile product used by the Cholesky / triangular-inverse steps
// (and as the fp32-exact fallback-free stepping stone for small problems).
//
// acc[TM][TN] += sum_{k in [k0,k1)} la(m0+m, k) * lb(k, n0+n)
// with thread-owned rows m = ty + i*(BM/TM) and cols n = tx + j*(BN/TN)
// (interleaved so that shared-memory reads are conflict-free).
#pragma once
#include <cuda_runtime.h>

namespace kfac {

template <int BM, int BN, int BK, int TM, int TN>
struct SimtTile {
  static constexpr int kThreads = (BM / TM) * (BN / TN);
  static constexpr int kLA = BK * BM / kThreads;  // A elements per thread per k-chunk
  static constexpr int kLB = BK * BN / kThreads;
  static constexpr int PA = BM + 1, PB = BN + 1;  // padded shared rows: conflict-free both ways
  static constexpr int kSmemFloats = 2 * BK * (PA + PB);   // double-buffered
  static_assert(BK * BM % kThreads == 0 && BK * BN % kThreads == 0, "even split of loads");

  // The next k-chunk is loaded into registers while the current one is being
  // multiplied out of shared memory (one barrier per chunk).  AK / BK_: the
  // operand is contiguous along k in global memory (row-major with k along the
  // row), so consecutive threads take consecutive k; otherwise consecutive
  // threads take consecutive rows (columns) of the operand.  Either way warps
  // read contiguous runs.
  template <bool AK = false, bool BKF = false, class LA, class LB>
  __device__ __forceinline__ static void run(const LA& la, const LB& lb, long long m0, long long n0,
                                             long long k0, long long k1, float (&acc)[TM][TN],
                                             float* smem) {
    const int tid = threadIdx.x;
    const int tx = tid % (BN / TN), ty = tid / (BN / TN);
    float ra[kLA], rb[kLB];
    auto a_pos = [&](int e, int* m, int* k) {
      if (AK) { *m = e / BK; *k = e % BK; } else { *m = e % BM; *k = e / BM; }
    };
    auto b_pos = [&](int e, int* c, int* k) {
      if (BKF) { *c = e / BK; *k = e % BK; } else { *c = e % BN; *k = e / BN; }
    };
    auto fetch = [&](long long kk) {
#pragma unroll
      for (int u = 0; u < kLA; ++u) {
        int m, k;
        a_pos(tid + u * kThreads, &m, &k);
        ra[u] = (kk + k < k1) ? la(m0 + m, kk + k) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kLB; ++u) {
        int c, k;
        b_pos(tid + u * kThreads, &c, &k);
        rb[u] = (kk + k < k1) ? lb(kk + k, n0 + c) : 0.f;
      }
    };
    if (k0 >= k1) return;
    fetch(k0);
    int buf = 0;
    for (long long kk = k0; kk < k1; kk += BK) {
      float* As = smem + buf * BK * (PA + PB);  // [BK][PA]
      float* Bs = As + BK * PA;                 // [BK][PB]
#pragma unroll
      for (int u = 0; u < kLA; ++u) {
        int m, k;
        a_pos(tid + u * kThreads, &m, &k);
        As[k * PA + m] = ra[u];
      }
#pragma unroll
      for (int u = 0; u < kLB; ++u) {
        int c, k;
        b_pos(tid + u * kThreads, &c, &k);
        Bs[k * PB + c] = rb[u];
      }
      __syncthreads();
      if (kk + BK < k1) fetch(kk + BK);
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[TM], b[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = As[k * PA + ty + i * (BM / TM)];
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = Bs[k * PB + tx + j * (BN / TN)];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      buf ^= 1;
    }
    __syncthreads();  // the caller may reuse smem after return
  }

  __device__ __forceinline__ static int row_of(int i) {
    return (threadIdx.x / (BN / TN)) + i * (BM / TM);
  }
  __device__ __forceinline__ static int col_of(int j) {
    return (threadIdx.x % (BN / TN)) + j * (BN / TN);
  }
};

// Strided fp32 operand: element (r, c) at p[r*rs + c*cs], zero outside [0,R) x [0,C).
struct StridedLoader {
  const float* p;
  long long rs, cs, R, C;
  __device__ __forceinline__ float operator()(long long r, long long c) const {
    return (r < R && c < C) ? p[r * rs + c * cs] : 0.f;
  }
};

}  // namespace kfac
