// Grouped symmetric rank-k update on CUDA cores: C <- beta C + alpha x-hat^T x-hat.
#pragma once
#include "kfac_internal.cuh"
#include "simt_gemm.cuh"

namespace kfac {

struct SyrkTile {
  static constexpr int BM = 128, BN = 128, BK = 8, TM = 8, TN = 8;
  using Tile = SimtTile<BM, BN, BK, TM, TN>;
};

// One symmetric product.  x is [M rows x d cols] row-major (ld); x-hat appends a
// ones column when has_bias (n = d + has_bias).  With x_lower, x is known to be
// lower triangular (x[r][c] = 0 for r < c) and rows below max(col) are skipped.
struct SyrkJob {
  const void* x;
  int64_t ld, M;
  int d, n, has_bias, x_lower;
  float alpha, beta;
  float* C;              // n x n, ld n; entries (r <= c) and mirrors written
  int nt;                // tiles per side
  int splits;            // split-K count (1: epilogue fused)
  int64_t rows_per_split;
  float* part;           // splits > 1: partial tiles [tiles][splits][BM*BN]
  int* tickets;          // splits > 1: one counter per tile, zero between launches
  int skip;              // grouped launches: job handled elsewhere (tensor-core path)
};

void syrk_split_plan(int n, int64_t rows, int* splits_out, int64_t* rows_per_split_out);

// Single job passed by value (factor update).
kfac_status launch_syrk_simt(const SyrkJob* job, int njobs_must_be_1, bool bf16, cudaStream_t st);
// Grouped jobs from a device table (inverse assembly); fp32 input, splits == 1.
kfac_status launch_syrk_simt_grouped(const SyrkJob* d_jobs, int njobs, int max_tiles,
                                     cudaStream_t st);

}  // namespace kfac
