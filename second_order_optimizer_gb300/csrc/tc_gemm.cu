// Tensor-core GEMM engine (tcgen05 + TMA) and the K1 factor update built on it.
//
//   C[M x N] = A[M x K] . B[N x K]^T, both operands K-major, fp32 accumulate,
//   with one of three fused epilogues:
//     SYRK     F <- beta F + alpha C on tiles on/above the diagonal, plus mirrors (K1,
//              with A = B = X = x-hat^T)
//     SPLIT    store C^T as TF32 halves (hi, lo), or as TF32 hi and bf16 correction
//              pairs (out_corr), ready to be the next product's operand; with no lo
//              buffer, alpha C^T as fp32 (or as bf16: out_bf16)
//     PRECOND  P^T = C; optional momentum / weight-decay / lr update of W in place (K4)
//
// Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
// Kronecker-Factored Approximate Curvature ...": §3.2 (A from activations, G from
// output gradients), §3.4 (Tensor Cores for the Kronecker-factor computation;
// a symmetric N x N factor has N(N+1)/2 distinct entries, so only tiles on or
// above the diagonal are computed and the epilogue writes each entry and its
// mirror).  CAFIN briefing, Introduction: EMA of the factors, fused into the
// epilogue as beta*F_old + alpha*acc.
//
// Two kernels:
//  pack:  x-hat [M x n] (row-major, any ld, fp32 or bf16, ones column virtual)
//         -> X = x-hat^T [n x Kp], K-major, so both MMA operands are K-major
//         tiles.  fp32 input is split into TF32 halves hi = rna(x),
//         lo = rna(x - hi) (3xTF32: hi*hi + hi*lo + lo*hi carries ~21 bits).
//         Operands with TcOperand::corr replace the two cross MMAs by one bf16
//         MMA over (hi, x - hi) pairs (tc::corr_pair; ~20 bits).
//  syrk:  one 128 x 128 output tile per CTA (split-K over rows when the
//         triangle has fewer tiles than SMs), warp-specialised:
//           warp 0  TMA producer   (SW128 tiles of 128 rows x 128 bytes)
//           warp 1  MMA issuer     (tcgen05.mma, accumulator in TMEM)
//           warps 2-9 epilogue     (tcgen05.ld; two warps per 32-lane TMEM quarter,
//                                   each holding half of the tile's columns)
//         The accumulator is double-buffered in TMEM and drained into fp32
//         registers every `ksub` rows, so no TMEM accumulation runs longer
//         than ksub rows whatever the tensor core's internal rounding.
//         Output goes through shared memory so both the tile and its mirror
//         are written with coalesced stores.
#include "kfac_internal.cuh"
#include "tc_prims.cuh"

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>

namespace kfac {

namespace {

template <bool kBF16, int BN_>
struct TcCfg {
  static constexpr int BM = 128, BN = BN_;         // UMMA 128 x BN per CTA (BN 128 or 256)
  static constexpr int R = BN / BM;                // B tile = R stacked A-sized tiles
  static constexpr int ELT = kBF16 ? 2 : 4;
  static constexpr int BK = 128 / ELT;            // k elements per 128-byte row
  static constexpr int KMMA = 32 / ELT;           // k elements per MMA (32 bytes)
  static constexpr int A_BYTES = BM * 128;        // A operand tile: 16 KB
  static constexpr int B_BYTES = BN * 128;        // B operand tile: 32 KB
  static constexpr int HALF_BYTES = A_BYTES + B_BYTES;           // hi (or bf16) part
  static constexpr int STAGE_BYTES = kBF16 ? HALF_BYTES : 2 * HALF_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES;   // 192 KB of stages
  static constexpr int TMEM_COLS = 2 * BN;        // double-buffered accumulator
  static constexpr int EPI_WARPS = 8;             // two per TMEM lane quarter
  static constexpr int CW = BN / 2;               // accumulator columns per epilogue thread
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int TPAD = BN + 1;             // output staging row pitch (floats)
  // After the main loop the stage buffers hold the output tile T [BM][TPAD] and,
  // behind it, the epilogue's global inputs (old F, or W and m) for RIN rows at a
  // time, fetched with asynchronous copies.
  static constexpr int T_BYTES = BM * TPAD * 4;
  static constexpr int RIN = BN == 128 ? 128 : 32;
  static constexpr int REGION = STAGES * STAGE_BYTES > T_BYTES + 2 * RIN * BN * 4
                                    ? STAGES * STAGE_BYTES
                                    : T_BYTES + 2 * RIN * BN * 4;
  static constexpr size_t SMEM = 1024 + (size_t)REGION + 256;
  static_assert(T_BYTES % 16 == 0, "input staging aligned");
};

struct GemmTcParams {
  int64_t M, N, K;
  int tiles_n;           // full grid: tile t -> (t / tiles_n, t % tiles_n)
  int upper;             // upper: only tiles reaching the upper triangle (SYRK, M == N)
  int tiles_m;           // tile rows (128 each)
  int same_ab;           // A and B are the same operand (diagonal tiles load once)
  int splits;            // k-splits per tile = csize x groups
  int csize;             // splits per thread-block cluster, reduced through DSMEM (1: none)
  int mc;                // cluster pairs share the B tile by TMA multicast (no split-K)
  int64_t k_per_split;   // multiple of ksub
  int kmode;             // reduction range per tile (TcProblem::kmode)
  int colmajor;          // persistent kernels: tiles column by column (grouped_tile)
  int ksub;              // k elements per TMEM drain (multiple of BK)
  int bias_col;          // MN-major pair SYRK: feature read from the ones map (or -1)
  int mn_full;           //   features in whole 64-feature chunks (64 floor(d / 64))
  int corr;              // fp32 operands in the TF32 + bf16-correction form (TcOperand::corr)
  float* part;           // this product's cluster partials [tile][groups][BM][BN]
  int* tickets;          // this product's tickets [tile][csize]
  DevStatus* status;
  int layer;
  TcEpilogue e;
};

// Tiles of 128 rows x (R*128) columns that reach the upper triangle: column block
// tj holds row blocks ti <= R tj + R - 1 (and ti < tiles_m); t enumerates them
// column by column.
__host__ __device__ inline int64_t upper_tile_count(int tiles_m, int tiles_n, int R) {
  int64_t c = 0;
  for (int tj = 0; tj < tiles_n; ++tj) c += (R * tj + R < tiles_m ? R * tj + R : tiles_m);
  return c;
}

// Multicast pairs: tiles column by column, each column's tile count padded to
// even so that a cluster pair (consecutive blocks) always shares the column tj
// (the B tile).  A padding slot computes its partner's tile and writes nothing.
__host__ __device__ inline int mc_column_tiles(int tiles_m, int R, bool upper, int tj) {
  const int c = upper ? (R * tj + R < tiles_m ? R * tj + R : tiles_m) : tiles_m;
  return c + (c & 1);
}
__host__ __device__ inline int64_t mc_tile_count(int tiles_m, int tiles_n, int R, bool upper) {
  int64_t c = 0;
  for (int tj = 0; tj < tiles_n; ++tj) c += mc_column_tiles(tiles_m, R, upper, tj);
  return c;
}
__device__ __forceinline__ void mc_tile(int t, int tiles_m, int tiles_n, int R, bool upper, int* ti,
                                        int* tj, bool* pad) {
  int j = 0;
  for (; j < tiles_n; ++j) {
    const int cp = mc_column_tiles(tiles_m, R, upper, j);
    if (t < cp) break;
    t -= cp;
  }
  const int cnt = upper ? (R * j + R < tiles_m ? R * j + R : tiles_m) : tiles_m;
  *pad = t >= cnt;
  *ti = *pad ? cnt - 1 : t;
  *tj = j;
}

__device__ __forceinline__ void upper_tile(int t, int tiles_m, int R, int* ti, int* tj) {
  int j = 0;
  for (;;) {
    const int cnt = R * j + R < tiles_m ? R * j + R : tiles_m;
    if (t < cnt) break;
    t -= cnt;
    ++j;
  }
  *ti = t;
  *tj = j;
}

// Reduction range of a tile whose columns start at c0 (width bn), for products
// with a triangular operand: kmode 0 the whole [0, K); 1 k >= c0 (the operand
// that carries the output column is zero for k below it, as a lower-triangular
// X in X^T X); 2 k < c0 + bn (zero for k past the column, as a lower-triangular
// right factor stored row-major).  c0 is a multiple of every k-block.
__host__ __device__ inline void k_range(int kmode, int64_t K, int64_t c0, int bn, int64_t* klo,
                                        int64_t* khi) {
  *klo = 0;
  *khi = K;
  if (kmode == 1) *klo = c0 < K ? c0 : K;
  else if (kmode == 2) *khi = c0 + bn < K ? c0 + bn : K;
}

// SPLIT output entry C^T[gc][gr] = v in the TF32 + bf16-correction form (an A
// operand of the next product): the TF32 hi in out_hi, the bf16 pair of
// tc::corr_pair in out_lo.
__device__ __forceinline__ void store_corr(const TcEpilogue& E, int64_t gc, int64_t gr, float v) {
  uint32_t pr;
  E.out_hi[gc * E.ldo + gr] = tc::corr_pair(v, false, &pr);
  reinterpret_cast<uint32_t*>(E.out_lo)[gc * E.ldo + gr] = pr;
}

// One output tile (and one k-split of it).
template <bool kBF16, int BN, int EPI>
__device__ __forceinline__ void gemm_body(const CUtensorMap* map_a_hi, const CUtensorMap* map_a_lo,
                                          const CUtensorMap* map_b_hi, const CUtensorMap* map_b_lo,
                                          const GemmTcParams& p, const int tile, const int split) {
  using C = TcCfg<kBF16, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::REGION);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int ti, tj;
  bool pad = false;   // multicast padding slot: computes, writes nothing
  const int mc_rank = p.mc ? (int)(blockIdx.x & 1) : 0;
  if (p.mc) {
    mc_tile(tile, p.tiles_m, p.tiles_n, C::R, p.upper != 0, &ti, &tj, &pad);
  } else if (p.upper) {
    upper_tile(tile, p.tiles_m, C::R, &ti, &tj);
  } else {
    ti = tile / p.tiles_n;
    tj = tile % p.tiles_n;
  }
  // A rows inside the B tile (same operand, ti / R == tj): read A out of B's smem
  const int a_in_b = (p.same_ab && ti / C::R == tj) ? ti % C::R + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], p.mc ? 2 : 1);   // multicast: both CTAs release a stage
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 32 * C::EPI_WARPS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(map_a_hi);
    tc::tma_prefetch_desc(map_b_hi);
    if (!kBF16) {
      tc::tma_prefetch_desc(map_a_lo);
      tc::tma_prefetch_desc(map_b_lo);
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  // multicast: the peer's barriers must be initialised before either CTA loads
  if (p.mc) cooperative_groups::this_cluster().sync();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // setup done: wait for the grids this one reads from, let the next one start
  pdl_wait();
  pdl_trigger();

  int64_t kbeg = (int64_t)split * p.k_per_split;
  int64_t kend = min(p.K, kbeg + p.k_per_split);
  {   // structurally zero parts of the reduction (triangular operands) are skipped
    int64_t klo, khi;
    k_range(p.kmode, p.K, (int64_t)tj * C::BN, C::BN, &klo, &khi);
    kbeg = max(kbeg, klo);
    kend = min(kend, khi);
  }
  const int nkb = kend > kbeg ? (int)((kend - kbeg + C::BK - 1) / C::BK) : 0;
  const int kb_per_sub = p.ksub / C::BK;
  const int nsub = (nkb + kb_per_sub - 1) / kb_per_sub;
  // stage layout: [A hi 16 KB][B hi 32 KB] ([A lo][B lo] for 3xTF32)
  auto a_ptr = [&](int s, int lo) {
    return smem + (size_t)s * C::STAGE_BYTES + lo * C::HALF_BYTES;
  };
  auto b_ptr = [&](int s, int lo) { return a_ptr(s, lo) + C::A_BYTES; };
  auto a_src = [&](int s, int lo) {  // where the MMA reads A from
    return a_in_b ? b_ptr(s, lo) + (a_in_b - 1) * C::A_BYTES : a_ptr(s, lo);
  };

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t bytes = (a_in_b ? C::B_BYTES : C::HALF_BYTES) * (kBF16 ? 1 : 2);
      // multicast: this CTA loads half of the B tile's rows into both CTAs
      const int b_off = mc_rank * (C::B_BYTES / 2), b_row = tj * C::BN + mc_rank * (C::BN / 2);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
          *abort_flag = 1;
          report_error(p.status, KFAC_ERR_TIMEOUT, p.layer, 1);
          break;
        }
        const int k0 = (int)(kbeg + (int64_t)kb * C::BK);
        tc::mbar_expect_tx(&full[stage], bytes);
        if (!a_in_b) tc::tma_load_2d(a_ptr(stage, 0), map_a_hi, &full[stage], k0, ti * C::BM);
        if (p.mc)
          tc::tma_load_2d_mc(b_ptr(stage, 0) + b_off, map_b_hi, &full[stage], k0, b_row, 3);
        else
          tc::tma_load_2d(b_ptr(stage, 0), map_b_hi, &full[stage], k0, tj * C::BN);
        if (!kBF16) {
          if (!a_in_b) tc::tma_load_2d(a_ptr(stage, 1), map_a_lo, &full[stage], k0, ti * C::BM);
          if (p.mc)
            tc::tma_load_2d_mc(b_ptr(stage, 1) + b_off, map_b_lo, &full[stage], k0, b_row, 3);
          else
            tc::tma_load_2d(b_ptr(stage, 1), map_b_lo, &full[stage], k0, tj * C::BN);
        }
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------ MMA issuer
      constexpr uint32_t idesc = tc::make_idesc(kBF16 ? 1 : 2, C::BM, C::BN);
      constexpr uint32_t idesc_c = tc::make_idesc(1, C::BM, C::BN);   // bf16 corrections
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int sub = 0; sub < nsub && ok; ++sub) {
        const int buf = sub & 1;
        if (!tc::mbar_wait(&acc_empty[buf], ((sub >> 1) & 1) ^ 1, abort_flag)) {
          report_error(p.status, KFAC_ERR_TIMEOUT, p.layer, 2);
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * C::BN);
        const int kb0 = sub * kb_per_sub, kb1 = min(nkb, kb0 + kb_per_sub);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
            report_error(p.status, KFAC_ERR_TIMEOUT, p.layer, 3);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_hi = tc::smem_u32(a_src(stage, 0));
          const uint32_t b_hi = tc::smem_u32(b_ptr(stage, 0));
          const uint32_t a_lo = tc::smem_u32(a_src(stage, kBF16 ? 0 : 1));
          const uint32_t b_lo = tc::smem_u32(b_ptr(stage, kBF16 ? 0 : 1));
#pragma unroll
          for (int kk = 0; kk < C::BK / C::KMMA; ++kk) {
            const uint32_t off = kk * 32;
            const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
            if (kBF16) {
              tc::umma_f16(d, tc::sdesc_kmajor_sw128(a_hi + off), tc::sdesc_kmajor_sw128(b_hi + off),
                           idesc, acc);
            } else if (p.corr) {
              tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                            tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
              tc::umma_f16(d, tc::sdesc_kmajor_sw128(a_lo + off),
                           tc::sdesc_kmajor_sw128(b_lo + off), idesc_c, 1u);
            } else {
              tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                            tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
              tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                            tc::sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
              tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_lo + off),
                            tc::sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
            }
          }
          if (p.mc)
            tc::umma_commit_mc(&empty[stage], 3);
          else
            tc::umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc::umma_commit(&acc_full[buf]);
      }
    }
  }

  // ------------------------------------------------------------ epilogue warps
  // Every epilogue writes C^T-oriented: the thread holding accumulator row gr
  // writes base[gc * ld + gr] for its columns gc, so consecutive lanes (rows)
  // store to consecutive addresses.  SYRK: that is the mirror F[gc][gr] (the
  // direct half F[gr][gc] goes through shared memory); SPLIT: X^T; PRECOND: the
  // product is computed transposed, C[j][i] = P[i][j], so W[i][j] = base[i d_in + j].
  float* T = reinterpret_cast<float*>(smem);  // [BM][TPAD], reuses the stage buffers
  // By value: p lives in kernel parameter space (indexed by problem in the grouped
  // kernel); read through a reference, every field would be reloaded after each
  // global store, which the compiler cannot prove does not alias it.
  const TcEpilogue E = p.e;
  const int64_t pM = p.M, pN = p.N;
  const int64_t r0 = (int64_t)ti * C::BM, c0 = (int64_t)tj * C::BN;
  // register path (no split-K, 128-wide tiles): results go to global memory from
  // the registers the accumulator was drained into
  const bool reg = C::BN == 128 && p.splits == 1;
  // global inputs of the register path, staged column-major ([BN][BM], lanes on
  // rows) behind T: SYRK old F; PRECOND W then m
  float* S = reinterpret_cast<float*>(smem + C::T_BYTES);
  static_assert(C::BN != 128 || C::T_BYTES + 2 * C::BN * C::BM * 4 <= C::REGION, "staging fits");
  if (warp >= 2) {
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;          // column half: [CW h, CW h + CW)
    const int row = 32 * q + lane;
    const int64_t gr = r0 + row;
    if (reg && gr < pM) {
      // Pull this thread's epilogue inputs into L2 while the main loop runs (it
      // feeds from L2, so HBM is idle); without this every CTA of a wave fetches
      // them from HBM in the same few microseconds at the end.
      if (EPI == TC_EPI_SYRK && E.beta != 0.f) {
        for (int c = 0; c < C::CW; ++c) {
          const int64_t gc = c0 + h * C::CW + c;
          if (gc < pN && gr <= gc) tc::prefetch_l2(E.C + gc * E.ldc + gr);
        }
      } else if (EPI == TC_EPI_PRECOND && E.pw && gr < E.d_in) {
        for (int c = 0; c < C::CW; ++c) {
          const int64_t i = c0 + h * C::CW + c;
          if (i >= pN) break;
          tc::prefetch_l2(E.pw + i * E.d_in + gr);
          tc::prefetch_l2(E.mw + i * E.d_in + gr);
        }
      }
    }
    float sum[C::CW];
#pragma unroll
    for (int c = 0; c < C::CW; ++c) sum[c] = 0.f;
    bool drained = true;
    for (int sub = 0; sub < nsub; ++sub) {
      const int buf = sub & 1;
      if (!tc::mbar_wait(&acc_full[buf], (sub >> 1) & 1, abort_flag)) {
        report_error(p.status, KFAC_ERR_TIMEOUT, p.layer, 4);
        *abort_flag = 1;
        drained = false;
        break;
      }
      tc::tc_fence_after();
      if (reg && sub == nsub - 1 && gr < pM && !pad) {
        // every MMA has completed: the stage buffers are free for the inputs
        if (EPI == TC_EPI_SYRK && E.beta != 0.f) {
#pragma unroll 8
          for (int c = 0; c < C::CW; ++c) {
            const int64_t gc = c0 + h * C::CW + c;
            if (gc < pN && gr <= gc)
              tc::cp_async4(S + (h * C::CW + c) * C::BM + row, E.C + gc * E.ldc + gr);
          }
        } else if (EPI == TC_EPI_PRECOND && E.pw) {
#pragma unroll 8
          for (int c = 0; c < C::CW; ++c) {
            const int64_t i = c0 + h * C::CW + c;
            if (i >= pN) continue;
            const int sidx = (h * C::CW + c) * C::BM + row;
            const bool wcol = gr < E.d_in;
            tc::cp_async4(S + sidx, wcol ? E.pw + i * E.d_in + gr : E.pb + i);
            tc::cp_async4(S + C::BN * C::BM + sidx, wcol ? E.mw + i * E.d_in + gr : E.mb + i);
          }
        }
      }
#pragma unroll
      for (int cc = 0; cc < C::CW / 32; ++cc) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) +
                          (uint32_t)(buf * C::BN + h * C::CW + cc * 32), v);
#pragma unroll
        for (int i = 0; i < 32; ++i) sum[cc * 32 + i] += v[i];
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&acc_empty[buf]);
    }
    if (reg && drained && gr < pM && !pad) {
      tc::cp_async_wait_all();   // this thread's own copies
      if (EPI == TC_EPI_SYRK) {
#pragma unroll
        for (int c = 0; c < C::CW; ++c) {
          const int64_t gc = c0 + h * C::CW + c;
          const bool ok = gc < pN && gr <= gc;
          const float old = (ok && E.beta != 0.f) ? S[(h * C::CW + c) * C::BM + row] : 0.f;
          const float v = fmaf(E.beta, old, E.alpha * sum[c]);
          sum[c] = v;
          if (ok) E.C[gc * E.ldc + gr] = v;
        }
      } else if (EPI == TC_EPI_SPLIT) {
        if (E.out_bf16) {   // alpha C^T as bf16
          __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(E.out_hi);
#pragma unroll
          for (int c = 0; c < C::CW; ++c) {
            const int64_t gc = c0 + h * C::CW + c;
            if (gc < pN) ob[gc * E.ldo + gr] = __float2bfloat16_rn(E.alpha * sum[c]);
          }
        } else if (E.out_lo && E.out_corr) {
#pragma unroll
          for (int c = 0; c < C::CW; ++c) {
            const int64_t gc = c0 + h * C::CW + c;
            if (gc < pN) store_corr(E, gc, gr, sum[c]);
          }
        } else if (E.out_lo) {
#pragma unroll
          for (int c = 0; c < C::CW; ++c) {
            const int64_t gc = c0 + h * C::CW + c;
            if (gc >= pN) continue;
            const float hi = tc::to_tf32(sum[c]);
            E.out_hi[gc * E.ldo + gr] = hi;
            E.out_lo[gc * E.ldo + gr] = tc::to_tf32(sum[c] - hi);
          }
        } else {   // alpha C^T (+ beta C_old^T) as fp32
#pragma unroll
          for (int c = 0; c < C::CW; ++c) {
            const int64_t gc = c0 + h * C::CW + c;
            if (gc >= pN) continue;
            float* o = E.out_hi + gc * E.ldo + gr;
            *o = E.beta != 0.f ? fmaf(E.beta, *o, E.alpha * sum[c]) : E.alpha * sum[c];
          }
        }
      } else {  // PRECOND: row gr = column j of P, column gc = row i
        const bool wcol = gr < E.d_in;
#pragma unroll
        for (int c = 0; c < C::CW; ++c) {
          const int64_t i = c0 + h * C::CW + c;
          if (i >= pN) continue;
          const int sidx = (h * C::CW + c) * C::BM + row;
          const float pr = sum[c];
          const float w = E.pw ? S[sidx] : 0.f;
          const float m = E.pw ? S[C::BN * C::BM + sidx] : 0.f;
          const float mn = fmaf(E.mu, m, fmaf(E.lambda, w, pr));
          const float wn = fmaf(-E.eta, mn, w);
          if (wcol) {
            const int64_t x = i * E.d_in + gr;
            if (E.ow) E.ow[x] = pr;
            if (E.pw) {
              E.mw[x] = mn;
              E.pw[x] = wn;
            }
          } else {
            if (E.ob) E.ob[i] = pr;
            if (E.pb) {
              E.mb[i] = mn;
              E.pb[i] = wn;
            }
          }
        }
      }
    }
    if (!reg || EPI == TC_EPI_SYRK) {
      // stage the tile for coalesced output (SYRK: the new values, for the direct half)
      asm volatile("bar.sync 1, %0;" ::"n"(32 * C::EPI_WARPS) : "memory");
#pragma unroll
      for (int c = 0; c < C::CW; ++c) T[row * C::TPAD + h * C::CW + c] = sum[c];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
  // multicast: every MMA of both CTAs has completed once both pass this point,
  // so no peer load or stage release can still land in this CTA's shared memory
  if (p.mc) {
    cooperative_groups::this_cluster().sync();
    if (pad) return;
  }
  constexpr int nth = C::THREADS;
  if (reg) {
    if (EPI == TC_EPI_SYRK && !*abort_flag) {
      // direct entries gr < gc from the staged new values, coalesced over gc
#pragma unroll 4
      for (int e = threadIdx.x; e < C::BM * C::BN; e += nth) {
        const int r = e / C::BN, c = e % C::BN;
        const int64_t gr = r0 + r, gc = c0 + c;
        if (gr < pM && gc < pN && gr < gc) E.C[gr * E.ldc + gc] = T[r * C::TPAD + c];
      }
    }
    return;
  }

  // Split-K: the tile's splits = csize x groups.  The csize splits of a cluster
  // sum their staged tiles through distributed shared memory, member c keeping
  // rows [row_lo, row_hi); with groups > 1 each member then writes its rows as a
  // cluster partial, and the last of the groups to arrive (a ticket per row
  // slice) sums the partials in group order and finishes those rows.  Fixed
  // order throughout, so results are deterministic.
  // Reduction loops run in batches of U elements per thread: all loads of a
  // batch are issued before any store.
  constexpr int NT = C::BM * C::BN;
  constexpr int U = 8;
  int row_lo = 0, row_hi = C::BM;   // rows of the tile this CTA finishes
  if (p.splits > 1) {
    const int CS = p.csize, G = p.splits / p.csize;
    int c = 0;
    if (CS > 1) {
      // Every member takes both cluster barriers, whatever happened before.
      namespace cg = cooperative_groups;
      cg::cluster_group cl = cg::this_cluster();
      cl.sync();
      c = (int)cl.block_rank();
      const int rb = (C::BM + CS - 1) / CS;
      row_lo = min(C::BM, c * rb);
      row_hi = min(C::BM, row_lo + rb);
      if (!*abort_flag) {
        const float* src[8];
        for (int q = 0; q < CS; ++q) src[q] = cl.map_shared_rank(T, q);
        const int n_el = (row_hi - row_lo) * C::BN;
        for (int b0 = threadIdx.x; b0 < n_el; b0 += nth * U) {
          float acc[U];
          int idx[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int e = b0 + u * nth;
            idx[u] = e < n_el ? (row_lo + e / C::BN) * C::TPAD + e % C::BN : 0;
            acc[u] = 0.f;
          }
          for (int q = 0; q < CS; ++q) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = src[q][idx[u]];
#pragma unroll
            for (int u = 0; u < U; ++u) acc[u] += v[u];
          }
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (b0 + u * nth < n_el) T[idx[u]] = acc[u];
        }
      }
      cl.sync();  // no member reads a peer's tile after this point
    }
    // An aborted CTA still takes its ticket, so the count stays consistent for
    // later launches (the result is already flagged as an error).
    const bool aborted = *abort_flag;
    if (G > 1) {
      const int gi = split / CS;
      const int n_el = (row_hi - row_lo) * C::BN, e0 = row_lo * C::BN;
      float* part = p.part + (size_t)tile * G * NT;
      for (int e = threadIdx.x; e < n_el; e += nth)
        part[(size_t)gi * NT + e0 + e] = T[(row_lo + e / C::BN) * C::TPAD + e % C::BN];
      __threadfence();
      __syncthreads();
      int* ticket = p.tickets + tile * CS + c;
      if (threadIdx.x == 0) *s_last = (atomicAdd(ticket, 1) == G - 1);
      __syncthreads();
      if (!*s_last) return;
      __threadfence();
      for (int b0 = threadIdx.x; b0 < n_el; b0 += nth * U) {
        float acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = b0 + u * nth;
          acc[u] = e < n_el ? __ldcg(part + e0 + e) : 0.f;
        }
        for (int q = 1; q < G; ++q) {
          float v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int e = b0 + u * nth;
            v[u] = e < n_el ? __ldcg(part + (size_t)q * NT + e0 + e) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) acc[u] += v[u];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = b0 + u * nth;
          if (e < n_el) T[(row_lo + e / C::BN) * C::TPAD + e % C::BN] = acc[u];
        }
      }
      if (threadIdx.x == 0) *ticket = 0;
    }
    if (aborted) return;
  } else if (*abort_flag) {
    return;
  }
  __syncthreads();
  // ---------------------------------------------- epilogue from the staged tile
  // (split-K, or 256-wide tiles).  Rows [row_lo, row_hi) of T; transposed stores
  // walk rows fastest (coalesced over gr); global inputs are fetched RC rows at a
  // time with asynchronous copies into S (behind T).
  const int nrows = row_hi - row_lo;
  if (EPI == TC_EPI_SYRK) {
    // tile entries (r <= c): F[r][c] = alpha*acc + beta*F[r][c]; T keeps the result
    constexpr int RC = (C::REGION - C::T_BYTES) / (C::BN * 4) < C::BM
                           ? (C::REGION - C::T_BYTES) / (C::BN * 4) : C::BM;
    for (int ca = row_lo; ca < row_hi; ca += RC) {
      const int cb = min(row_hi, ca + RC);
      const int ne = (cb - ca) * C::BN;
      if (E.beta != 0.f) {
#pragma unroll 4
        for (int e = threadIdx.x; e < ne; e += nth) {
          const int64_t gr = r0 + ca + e / C::BN, gc = c0 + e % C::BN;
          if (gr < pM && gc < pN && gr <= gc) tc::cp_async4(S + e, E.C + gr * E.ldc + gc);
        }
        tc::cp_async_wait_all();
        __syncthreads();
      }
#pragma unroll 4
      for (int e = threadIdx.x; e < ne; e += nth) {
        const int r = ca + e / C::BN, c = e % C::BN;
        const int64_t gr = r0 + r, gc = c0 + c;
        if (!(gr < pM && gc < pN && gr <= gc)) continue;
        const float old = E.beta != 0.f ? S[e] : 0.f;
        const float v = fmaf(E.beta, old, E.alpha * T[r * C::TPAD + c]);
        E.C[gr * E.ldc + gc] = v;
        T[r * C::TPAD + c] = v;
      }
      __syncthreads();
    }
    // mirrors (gr < gc): F[gc][gr], coalesced over gr
#pragma unroll 4
    for (int e = threadIdx.x; e < nrows * C::BN; e += nth) {
      const int c = e / nrows, r = row_lo + e % nrows;
      const int64_t gr = r0 + r, gc = c0 + c;
      if (gr >= pM || gc >= pN || gr >= gc) continue;
      E.C[gc * E.ldc + gr] = T[r * C::TPAD + c];
    }
  } else if (EPI == TC_EPI_SPLIT) {
#pragma unroll 4
    for (int e = threadIdx.x; e < nrows * C::BN; e += nth) {
      const int c = e / nrows, r = row_lo + e % nrows;
      const int64_t gr = r0 + r, gc = c0 + c;
      if (gr >= pM || gc >= pN) continue;
      const float v = T[r * C::TPAD + c];
      if (E.out_bf16) {   // alpha C^T as bf16
        reinterpret_cast<__nv_bfloat16*>(E.out_hi)[gc * E.ldo + gr] = __float2bfloat16_rn(E.alpha * v);
        continue;
      }
      if (!E.out_lo) {   // alpha C^T (+ beta C_old^T) as fp32
        float* o = E.out_hi + gc * E.ldo + gr;
        *o = E.beta != 0.f ? fmaf(E.beta, *o, E.alpha * v) : E.alpha * v;
        continue;
      }
      if (E.out_corr) {
        store_corr(E, gc, gr, v);
        continue;
      }
      const float hi = tc::to_tf32(v);
      E.out_hi[gc * E.ldo + gr] = hi;
      E.out_lo[gc * E.ldo + gr] = tc::to_tf32(v - hi);
    }
  } else {  // TC_EPI_PRECOND: tile row gr = column j of P (j >= d_in: bias), column gc = row i
    constexpr int RC = (C::REGION - C::T_BYTES) / (2 * C::BN * 4) < C::BM
                           ? (C::REGION - C::T_BYTES) / (2 * C::BN * 4) : C::BM;
    float* Sw = S;
    float* Sm = S + RC * C::BN;
    for (int ca = row_lo; ca < row_hi; ca += RC) {
      const int cb = min(row_hi, ca + RC);
      const int nr = cb - ca;
      const int ne = nr * C::BN;
      if (E.pw) {
#pragma unroll 4
        for (int e = threadIdx.x; e < ne; e += nth) {
          const int64_t j = r0 + ca + e % nr, i = c0 + e / nr;
          if (!(j < pM && i < pN)) continue;
          if (j < E.d_in) {
            tc::cp_async4(Sw + e, E.pw + i * E.d_in + j);
            tc::cp_async4(Sm + e, E.mw + i * E.d_in + j);
          } else {
            tc::cp_async4(Sw + e, E.pb + i);
            tc::cp_async4(Sm + e, E.mb + i);
          }
        }
        tc::cp_async_wait_all();
        __syncthreads();
      }
#pragma unroll 4
      for (int e = threadIdx.x; e < ne; e += nth) {
        const int r = ca + e % nr, c = e / nr;
        const int64_t j = r0 + r, i = c0 + c;
        if (!(j < pM && i < pN)) continue;
        const float w = E.pw ? Sw[e] : 0.f, m = E.pw ? Sm[e] : 0.f;
        const float pr = T[r * C::TPAD + c];
        const float mn = fmaf(E.mu, m, fmaf(E.lambda, w, pr));
        const float wn = fmaf(-E.eta, mn, w);
        if (j < E.d_in) {
          const int64_t x = i * E.d_in + j;
          if (E.ow) E.ow[x] = pr;
          if (E.pw) {
            E.mw[x] = mn;
            E.pw[x] = wn;
          }
        } else {
          if (E.ob) E.ob[i] = pr;
          if (E.pb) {
            E.mb[i] = mn;
            E.pb[i] = wn;
          }
        }
      }
      __syncthreads();
    }
  }
}

template <bool kBF16, int BN, int EPI>
__global__ void __launch_bounds__(TcCfg<kBF16, BN>::THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a_hi,
               const __grid_constant__ CUtensorMap map_a_lo,
               const __grid_constant__ CUtensorMap map_b_hi,
               const __grid_constant__ CUtensorMap map_b_lo, const __grid_constant__ GemmTcParams p) {
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  gemm_body<kBF16, BN, EPI>(&map_a_hi, &map_a_lo, &map_b_hi, &map_b_lo, p, tile, split);
}

// Several independent products in one launch (128 x 128 tiles): blocks are laid
// out problem by problem, each problem's `splits` consecutive blocks per tile
// (csize of them form one cluster; csize is the same for the whole launch).
constexpr int kMaxGroup = 16;
struct GroupedTc {
  CUtensorMap maps[4 * kMaxGroup];  // per problem: A hi, A lo, B hi, B lo
  GemmTcParams prob[kMaxGroup];
  int block_start[kMaxGroup + 1];
  int count;
  int csize;
};

template <bool kBF16, int EPI>
__global__ void __launch_bounds__(TcCfg<kBF16, 128>::THREADS, 1)
gemm_tc_grouped_kernel(const __grid_constant__ GroupedTc g) {
  int q = 0;
  while (q + 1 < g.count && (int)blockIdx.x >= g.block_start[q + 1]) ++q;
  const int local = (int)blockIdx.x - g.block_start[q], sp = g.prob[q].splits;
  gemm_body<kBF16, 128, EPI>(&g.maps[4 * q], &g.maps[4 * q + 1], &g.maps[4 * q + 2],
                             &g.maps[4 * q + 3], g.prob[q], local / sp, local % sp);
}

// ------------------------------------------------------- persistent grouped
// The grouped products without split-K, one CTA per SM looping over tiles
// (tile t, t + gridDim.x, ...).  The TMA and MMA warps run on into the next
// tile while the drain warps finish the previous tile's epilogue: the TMEM
// accumulator is a ring of 512 columns (4 buffers of 128 x 128, or 2 of 128 x 256),
// so the MMA can run up to that many drain periods ahead.  The stage buffers
// stay busy meanwhile, so these epilogues read their global inputs straight
// into registers (lanes on rows, coalesced; prefetched into L2 when the tile
// starts) and the SYRK direct half is transposed through a per-warp buffer.
// Each drain thread holds 64 accumulator columns of one row: 8 drain warps for
// 128-wide tiles, 16 for 256-wide ones (four per TMEM lane quarter).
template <bool kBF16, int BN>
struct PersistCfg {
  using C = TcCfg<kBF16, BN>;                       // operand tiles: A 128 rows, B BN rows
  static constexpr int R = BN / 128;
  static constexpr int EPI_WARPS = BN / 16;         // 4 per 64 columns
  static constexpr int CW = 64;                     // accumulator columns per drain thread
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int ACC = 512 / BN;              // TMEM ring: 512 columns
  static constexpr int TMEM_COLS = ACC * BN;
  static constexpr int XW = BN == 128 ? 32 : 8;     // columns per transpose chunk
  static constexpr int XP = XW + 1;                 // transpose pitch
  static constexpr int XPOSE_BYTES = EPI_WARPS * 32 * XP * 4;
  static constexpr int FIT = (232448 - 1024 - 256 - XPOSE_BYTES) / C::STAGE_BYTES;
  static constexpr int STAGES = FIT < C::STAGES ? FIT : C::STAGES;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * C::STAGE_BYTES + XPOSE_BYTES + 256;
  static_assert(STAGES >= 2, "at least double-buffered operand stages");
  static_assert(SMEM <= 232448, "fits the per-CTA shared memory");
};

// Tile order of the persistent kernels, so that the tiles running at the same time
// (about one per SM) read each operand block from DRAM once and from L2 after.
// Upper-triangle (SYRK) products: blocks of kTileBlock x kTileBlock tiles, block
// columns in turn, tile columns inside a block.  Other products: along the
// longer side of the output, so that the larger operand is read once per launch
// and the smaller one is re-read (colmajor when M < N).
constexpr int kTileBlock = 8;
__host__ __device__ inline void upper_tile_blocked(int t, int tiles_m, int tiles_n, int* ti,
                                                   int* tj) {
  constexpr int S = kTileBlock;
  const int nbj = (tiles_n + S - 1) / S;
  for (int bj = 0; bj < nbj; ++bj) {
    const int c0 = bj * S, c1 = c0 + S < tiles_n ? c0 + S : tiles_n;
    for (int bi = 0; bi <= bj; ++bi) {
      const int r0 = bi * S;
      if (r0 >= tiles_m) break;
      const int r1 = r0 + S < tiles_m ? r0 + S : tiles_m;
      for (int c = c0; c < c1; ++c) {   // rows r0 <= r < min(r1, c + 1) of column c
        const int hi = c + 1 < r1 ? c + 1 : r1;
        const int k = hi > r0 ? hi - r0 : 0;
        if (t < k) {
          *ti = r0 + t;
          *tj = c;
          return;
        }
        t -= k;
      }
    }
  }
  *ti = *tj = 0;   // t beyond the triangle: not reached
}

template <int R>
__device__ __forceinline__ void grouped_tile(const GroupedTc& g, int t, int* q, int* ti, int* tj) {
  int k = 0;
  while (k + 1 < g.count && t >= g.block_start[k + 1]) ++k;
  const int local = t - g.block_start[k];
  const GemmTcParams& p = g.prob[k];
  if (p.upper) {
    if (R == 1)
      upper_tile_blocked(local, p.tiles_m, p.tiles_n, ti, tj);
    else
      upper_tile(local, p.tiles_m, R, ti, tj);
  } else if (p.colmajor) {
    *ti = local % p.tiles_m;
    *tj = local / p.tiles_m;
  } else {
    *ti = local / p.tiles_n;
    *tj = local % p.tiles_n;
  }
  *q = k;
}

// Start of a drained tile's running sum.  SYRK with an EMA (beta != 0) starts from
// the old factor value, read from where the epilogue will write it (the mirror
// half, row gc, column gr <= gc), so that the loads run while the tile's first
// partial accumulates and the epilogue has none.  With |alpha| <= |beta| the sum
// starts at C_old and takes each drained partial times alpha / beta (epilogue
// scale beta); otherwise it starts at (beta / alpha) C_old and takes the partials
// as they are (epilogue scale alpha): either way the scaled sum is
// beta C_old + alpha S, and no factor above 1 can overflow.  Returns the
// partials' scale; *oscale is the epilogue's.
template <int EPI, int CW>
__device__ __forceinline__ float sum_init(const TcEpilogue& E, float (&sum)[CW], int64_t c0,
                                          int64_t gr, int64_t pM, int64_t pN, float* oscale) {
  if (EPI == TC_EPI_SYRK && E.beta != 0.f) {
    const bool by_beta = fabsf(E.alpha) <= fabsf(E.beta);
    const float r = by_beta ? 1.f : E.beta / E.alpha;
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      const int64_t gc = c0 + c;
      sum[c] = (gr < pM && gc < pN && gr <= gc) ? __ldcg(E.C + gc * E.ldc + gr) : 0.f;
    }
    if (!by_beta) {
#pragma unroll
      for (int c = 0; c < CW; ++c) sum[c] *= r;
    }
    *oscale = by_beta ? E.beta : E.alpha;
    return by_beta ? E.alpha / E.beta : 1.f;
  }
#pragma unroll
  for (int c = 0; c < CW; ++c) sum[c] = 0.f;
  *oscale = E.alpha;
  return 1.f;
}

// Epilogue of a drained tile from registers (the persistent kernels): this thread
// holds accumulator row gr for the CW columns from c0.  Every store runs along
// rows across the warp (C^T-oriented), except the SYRK direct half, which goes
// through the warp's transpose buffer xb (32 rows x XW columns at a time).  EB
// global loads are kept in flight.
template <int EPI, int CW, int XW, int EB>
__device__ __forceinline__ void epilogue_from_registers(const TcEpilogue& E, float (&sum)[CW],
                                                        float* xb, int lane, int qd, int64_t r0,
                                                        int64_t c0, int64_t gr, int64_t pM,
                                                        int64_t pN, float oscale) {
  constexpr int XP = XW + 1;
  if (EPI == TC_EPI_SYRK) {
    // mirror F[gc][gr]: oscale * (the running sum started by sum_init)
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      const int64_t gc = c0 + c;
      const float v = oscale * sum[c];
      sum[c] = v;
      if (gr < pM && gc < pN && gr <= gc) E.C[gc * E.ldc + gr] = v;
    }
  }
  if (EPI == TC_EPI_SYRK) {
    // direct half F[gr][gc] (gr < gc): blocks of 32 rows x XW columns turned
    // through the warp's buffer so that lanes run along gc
    constexpr int RPI = 32 / XW;   // rows per store instruction
#pragma unroll
    for (int j2 = 0; j2 < CW / XW; ++j2) {
#pragma unroll
      for (int c = 0; c < XW; ++c) xb[lane * XP + c] = sum[j2 * XW + c];
      __syncwarp();
      const int cl = lane % XW;
      const int64_t gcol = c0 + j2 * XW + cl;
#pragma unroll 8
      for (int it = 0; it < 32 / RPI; ++it) {
        const int r = it * RPI + lane / XW;
        const int64_t grr = r0 + 32 * qd + r;
        if (grr < pM && gcol < pN && grr < gcol) E.C[grr * E.ldc + gcol] = xb[r * XP + cl];
      }
      __syncwarp();
    }
  } else if (EPI == TC_EPI_SPLIT) {
    if (gr < pM && E.out_bf16) {   // alpha C^T as bf16
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(E.out_hi);
#pragma unroll
      for (int c = 0; c < CW; ++c) {
        const int64_t gc = c0 + c;
        if (gc < pN) ob[gc * E.ldo + gr] = __float2bfloat16_rn(E.alpha * sum[c]);
      }
    } else if (gr < pM && E.out_lo && E.out_corr) {
#pragma unroll
      for (int c = 0; c < CW; ++c)
        if (c0 + c < pN) store_corr(E, c0 + c, gr, sum[c]);
    } else if (gr < pM && E.out_lo) {
#pragma unroll
      for (int c = 0; c < CW; ++c) {
        const int64_t gc = c0 + c;
        if (gc >= pN) continue;
        const float hi = tc::to_tf32(sum[c]);
        E.out_hi[gc * E.ldo + gr] = hi;
        E.out_lo[gc * E.ldo + gr] = tc::to_tf32(sum[c] - hi);
      }
    } else if (gr < pM) {   // alpha C^T (+ beta C_old^T) as fp32
#pragma unroll
      for (int c = 0; c < CW; ++c) {
        const int64_t gc = c0 + c;
        if (gc >= pN) continue;
        float* o = E.out_hi + gc * E.ldo + gr;
        *o = E.beta != 0.f ? fmaf(E.beta, *o, E.alpha * sum[c]) : E.alpha * sum[c];
      }
    }
  } else {  // PRECOND: row gr = column j of P, column gc = row i
    const bool wcol = gr < E.d_in;
    if (gr < pM) {
#pragma unroll
      for (int cc = 0; cc < CW; cc += EB) {
        float w[EB], m[EB];
#pragma unroll
        for (int u = 0; u < EB; ++u) {
          const int64_t i = c0 + cc + u;
          w[u] = m[u] = 0.f;
          if (E.pw && i < pN) {
            w[u] = wcol ? __ldcg(E.pw + i * E.d_in + gr) : __ldcg(E.pb + i);
            m[u] = wcol ? __ldcg(E.mw + i * E.d_in + gr) : __ldcg(E.mb + i);
          }
        }
#pragma unroll
        for (int u = 0; u < EB; ++u) {
          const int64_t i = c0 + cc + u;
          if (i >= pN) continue;
          const float pr = sum[cc + u];
          const float mn = fmaf(E.mu, m[u], fmaf(E.lambda, w[u], pr));
          const float wn = fmaf(-E.eta, mn, w[u]);
          if (wcol) {
            const int64_t x = i * E.d_in + gr;
            if (E.ow) E.ow[x] = pr;
            if (E.pw) {
              E.mw[x] = mn;
              E.pw[x] = wn;
            }
          } else {
            if (E.ob) E.ob[i] = pr;
            if (E.pb) {
              E.mb[i] = mn;
              E.pb[i] = wn;
            }
          }
        }
      }
    }
  }

}

template <bool kBF16, int EPI, int BN>
__device__ __forceinline__ void persistent_body(const GroupedTc& g) {
  using PC = PersistCfg<kBF16, BN>;
  using C = typename PC::C;
  constexpr int CW = PC::CW;
  constexpr int STAGES = PC::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + PC::XPOSE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + PC::ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + PC::ACC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int total = g.block_start[g.count];

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < PC::ACC; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 32 * PC::EPI_WARPS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, PC::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  auto a_ptr = [&](int s, int lo) { return smem + (size_t)s * C::STAGE_BYTES + lo * C::HALF_BYTES; };
  auto b_ptr = [&](int s, int lo) { return a_ptr(s, lo) + C::A_BYTES; };
  // k-blocks of tile (q, tj): [kb_lo, kb_lo + nkb) (TcProblem::kmode)
  auto kblocks = [&](int q, int tj, int* kb_lo) {
    int64_t klo, khi;
    k_range(g.prob[q].kmode, g.prob[q].K, (int64_t)tj * BN, BN, &klo, &khi);
    *kb_lo = (int)(klo / C::BK);
    return khi > klo ? (int)((khi - klo + C::BK - 1) / C::BK) : 0;
  };
  // same operand and the A rows inside the B tile: read A out of B's shared memory
  auto a_in_b = [&](int q, int ti, int tj) {
    return (g.prob[q].same_ab && ti / PC::R == tj) ? ti % PC::R + 1 : 0;
  };
  const int kb_per_sub = g.prob[0].ksub / C::BK;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int q, ti, tj;
        grouped_tile<PC::R>(g, t, &q, &ti, &tj);
        const CUtensorMap* m = &g.maps[4 * q];
        const int aib = a_in_b(q, ti, tj);
        const uint32_t bytes = (aib ? C::B_BYTES : C::HALF_BYTES) * (kBF16 ? 1 : 2);
        int kb_lo;
        const int nkb = kblocks(q, tj, &kb_lo);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            *abort_flag = 1;
            report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 11);
            ok = false;
            break;
          }
          const int k0 = (kb_lo + kb) * C::BK;
          tc::mbar_expect_tx(&full[stage], bytes);
          if (!aib) tc::tma_load_2d(a_ptr(stage, 0), &m[0], &full[stage], k0, ti * C::BM);
          tc::tma_load_2d(b_ptr(stage, 0), &m[2], &full[stage], k0, tj * BN);
          if (!kBF16) {
            if (!aib) tc::tma_load_2d(a_ptr(stage, 1), &m[1], &full[stage], k0, ti * C::BM);
            tc::tma_load_2d(b_ptr(stage, 1), &m[3], &full[stage], k0, tj * BN);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------ MMA issuer
      constexpr uint32_t idesc = tc::make_idesc(kBF16 ? 1 : 2, C::BM, BN);
      constexpr uint32_t idesc_c = tc::make_idesc(1, C::BM, BN);   // bf16 corrections
      int stage = 0;
      uint32_t phase = 0;
      int gsub = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int q, ti, tj;
        grouped_tile<PC::R>(g, t, &q, &ti, &tj);
        const int aib = a_in_b(q, ti, tj);
        const bool corr = !kBF16 && g.prob[q].corr != 0;
        int kb_lo;
        const int nkb = kblocks(q, tj, &kb_lo);
        const int nsub = (nkb + kb_per_sub - 1) / kb_per_sub;
        for (int sub = 0; sub < nsub && ok; ++sub, ++gsub) {
          const int buf = gsub % PC::ACC, use = gsub / PC::ACC;
          if (!tc::mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag)) {
            report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 12);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * BN);
          const int kb0 = sub * kb_per_sub, kb1 = min(nkb, kb0 + kb_per_sub);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
              report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 13);
              *abort_flag = 1;
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const int lo1 = kBF16 ? 0 : 1;
            const uint32_t a_hi = tc::smem_u32(aib ? b_ptr(stage, 0) + (aib - 1) * C::A_BYTES
                                                   : a_ptr(stage, 0));
            const uint32_t b_hi = tc::smem_u32(b_ptr(stage, 0));
            const uint32_t a_lo = tc::smem_u32(aib ? b_ptr(stage, lo1) + (aib - 1) * C::A_BYTES
                                                   : a_ptr(stage, lo1));
            const uint32_t b_lo = tc::smem_u32(b_ptr(stage, lo1));
#pragma unroll
            for (int kk = 0; kk < C::BK / C::KMMA; ++kk) {
              const uint32_t off = kk * 32;
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              if (kBF16) {
                tc::umma_f16(d, tc::sdesc_kmajor_sw128(a_hi + off),
                             tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
              } else if (corr) {
                tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                              tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
                tc::umma_f16(d, tc::sdesc_kmajor_sw128(a_lo + off),
                             tc::sdesc_kmajor_sw128(b_lo + off), idesc_c, 1u);
              } else {
                tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                              tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
                tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_hi + off),
                              tc::sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
                tc::umma_tf32(d, tc::sdesc_kmajor_sw128(a_lo + off),
                              tc::sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
              }
            }
            tc::umma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (ok) tc::umma_commit(&acc_full[buf]);
        }
      }
    }
  } else {  // ------------------------------------------------ drain + epilogue
    const int qd = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;           // column block: [CW h, CW h + CW)
    const int row = 32 * qd + lane;
    float* xb = xbuf + (warp - 2) * 32 * PC::XP;
    int gsub = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int q, ti, tj;
      grouped_tile<PC::R>(g, t, &q, &ti, &tj);
      const TcEpilogue E = g.prob[q].e;   // by value (see gemm_body)
      const int64_t pM = g.prob[q].M, pN = g.prob[q].N;
      const int64_t r0 = (int64_t)ti * C::BM, c0 = (int64_t)tj * BN + h * CW;
      const int64_t gr = r0 + row;
      int kb_lo;
      const int nkb = kblocks(q, tj, &kb_lo);
      const int nsub = (nkb + kb_per_sub - 1) / kb_per_sub;
      if (gr < pM) {   // the tile's epilogue inputs into L2 while the drains run
        if (EPI == TC_EPI_PRECOND && E.pw && gr < E.d_in) {
          for (int c = 0; c < CW; ++c) {
            const int64_t i = c0 + c;
            if (i >= pN) break;
            tc::prefetch_l2(E.pw + i * E.d_in + gr);
            tc::prefetch_l2(E.mw + i * E.d_in + gr);
          }
        }
      }
      float sum[CW];
      float oscale;
      const float kin = sum_init<EPI, CW>(E, sum, c0, gr, pM, pN, &oscale);
      for (int sub = 0; sub < nsub; ++sub, ++gsub) {
        const int buf = gsub % PC::ACC, use = gsub / PC::ACC;
        if (!tc::mbar_wait(&acc_full[buf], use & 1, abort_flag)) {
          report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 14);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc::tc_fence_after();
        if (BN == 128) {
#pragma unroll
          for (int cc = 0; cc < CW / 32; ++cc) {
            float v[32];
            tc::tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) +
                              (uint32_t)(buf * BN + h * CW + cc * 32), v);
#pragma unroll
            for (int i = 0; i < 32; ++i) sum[cc * 32 + i] = fmaf(kin, v[i], sum[cc * 32 + i]);
          }
        } else {   // fewer registers per drain thread (16 drain warps)
#pragma unroll
          for (int cc = 0; cc < CW / 16; ++cc) {
            float v[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) +
                              (uint32_t)(buf * BN + h * CW + cc * 16), v);
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[cc * 16 + i] = fmaf(kin, v[i], sum[cc * 16 + i]);
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&acc_empty[buf]);
      }
      if (!ok) break;
      epilogue_from_registers<EPI, CW, PC::XW, BN == 128 ? 16 : 8>(E, sum, xb, lane, qd, r0, c0, gr,
                                                                   pM, pN, oscale);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, PC::TMEM_COLS);
}

// 128-wide tiles: 320 threads; 256-wide tiles: 576 threads (18 warps, so two of
// the four SM sub-partitions hold five warps of their 16384 registers: at most
// 102 registers a thread, 96 in steps of 8).
template <bool kBF16, int EPI>
__global__ void __launch_bounds__(PersistCfg<kBF16, 128>::THREADS, 1)
gemm_tc_persistent_kernel(const __grid_constant__ GroupedTc g) {
  persistent_body<kBF16, EPI, 128>(g);
}
template <bool kBF16, int EPI>
__global__ void __maxnreg__(96) gemm_tc_persistent_wide_kernel(const __grid_constant__ GroupedTc g) {
  persistent_body<kBF16, EPI, 256>(g);
}
template <bool kBF16, int EPI, int BN>
struct PersistKernel {
  static constexpr auto fn = gemm_tc_persistent_kernel<kBF16, EPI>;
};
template <bool kBF16, int EPI>
struct PersistKernel<kBF16, EPI, 256> {
  static constexpr auto fn = gemm_tc_persistent_wide_kernel<kBF16, EPI>;
};

// ------------------------------------------------------- CTA-pair persistent
// Products with a wave of 256 x 256 tiles: clusters of two CTAs share each MMA
// (tcgen05 cta_group::2): a tile's 256 rows are 128 in each CTA's shared memory
// and TMEM, and each CTA loads half of the tile's 256 B rows, which the pair's
// MMA reads from both.  Per SM that is half the B operand traffic of a
// single-CTA 128 x 256 tile (TMA writes and MMA reads of shared memory).
//   both CTAs  warp 0      TMA producer: its A rows and its half of B, completing
//                          on the even CTA's stage barrier (cta_group::2 loads)
//   even CTA   warp 1      MMA issuer; commits release both CTAs' stages and
//                          signal both CTAs' accumulator barriers
//   both CTAs  warps 2-17  drain + epilogue of the CTA's 128 rows (as the
//                          single-CTA persistent kernel), one arrival per warp on
//                          the even CTA's accumulator-empty barrier
// The pair loops over tiles t = pair, pair + pairs, ...; every wait is bounded.
// kMN (the in-place bf16 SYRK): stages of 128 k rows, so that each operand's
// stage is one 32 KB box; 64-row stages (two boxes of 16 KB per stage and
// operand, six stages) ran the transformer factor phase 8% slower.
template <bool kBF16, bool kMN = false>
struct PairCfg {
  static constexpr int BM = 128, BN = 256;           // per CTA: 128 rows x 256 columns
  static constexpr int ELT = kBF16 ? 2 : 4;
  static constexpr int BK = kMN ? 128 : 128 / ELT;
  static constexpr int KMMA = 32 / ELT;
  static constexpr int A_BYTES = BM * BK * ELT;      // K-major: 128-byte rows, 16 KB
  static constexpr int BH_BYTES = (BN / 2) * BK * ELT;   // this CTA's half of B
  static constexpr int MN_CHUNK = BK * 128;          // MN-major: 64 features x BK k
  static constexpr int HALF_BYTES = A_BYTES + BH_BYTES;
  static constexpr int STAGE_BYTES = kBF16 ? HALF_BYTES : 2 * HALF_BYTES;
  static constexpr int EPI_WARPS = 16, CW = 64;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int ACC = 2, TMEM_COLS = 512;
  static constexpr int XW = 8, XP = 9;
  static constexpr int XPOSE_BYTES = EPI_WARPS * 32 * XP * 4;
  static constexpr int FIT = (232448 - 1024 - 512 - XPOSE_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = FIT < 6 ? FIT : 6;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + XPOSE_BYTES + 512;
  static_assert(STAGES >= 3, "operand stages");
  static_assert(SMEM <= 232448, "fits the per-CTA shared memory");
};

template <bool kBF16, int EPI, bool kMN>
__device__ __forceinline__ void pair_body(const GroupedTc& g) {
  using PC = PairCfg<kBF16, kMN>;
  static_assert(!kMN || (kBF16 && EPI == TC_EPI_SYRK), "MN-major operands: bf16 SYRK");
  constexpr int CW = PC::CW, BN = PC::BN, STAGES = PC::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * PC::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * PC::STAGE_BYTES + PC::XPOSE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + PC::ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + PC::ACC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int total = g.block_start[g.count];
  const uint32_t rank = tc::cluster_rank();
  const int pair = (int)(blockIdx.x / 2), npairs = (int)(gridDim.x / 2);
  // a role that gives up stops the peer CTA's roles too
  const uint32_t peer_abort = tc::mapa((const void*)abort_flag, rank ^ 1u);
  auto give_up = [&]() {
    *abort_flag = 1;
    tc::st_cluster_u32(peer_abort, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < PC::ACC; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 2 * PC::EPI_WARPS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tmem_slot, PC::TMEM_COLS);
    tc::tmem_relinquish_pair();
  }
  tc::tc_fence_before();
  __syncwarp();
  tc::cluster_sync();   // both CTAs' barriers initialised and TMEM allocated
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  auto a_ptr = [&](int s, int lo) { return smem + (size_t)s * PC::STAGE_BYTES + lo * PC::HALF_BYTES; };
  auto b_ptr = [&](int s, int lo) { return a_ptr(s, lo) + PC::A_BYTES; };
  auto kblocks = [&](int q, int tj, int* kb_lo) {
    int64_t klo, khi;
    k_range(g.prob[q].kmode, g.prob[q].K, (int64_t)tj * BN, BN, &klo, &khi);
    *kb_lo = (int)(klo / PC::BK);
    return khi > klo ? (int)((khi - klo + PC::BK - 1) / PC::BK) : 0;
  };
  // same operand, diagonal tile: this CTA's A rows are its half of B
  auto a_in_b = [&](int q, int ti, int tj) { return g.prob[q].same_ab && ti == tj; };
  const int kb_per_sub = g.prob[0].ksub / PC::BK;

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------ TMA producer
      const uint32_t full0 = tc::mapa(full, 0);   // the even CTA's stage barriers
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        int q, ti, tj;
        grouped_tile<1>(g, t, &q, &ti, &tj);
        const CUtensorMap* m = &g.maps[4 * q];
        const bool aib = a_in_b(q, ti, tj);
        const uint32_t bytes = (aib ? PC::BH_BYTES : PC::HALF_BYTES) * (kBF16 ? 1 : 2);
        const int arow = ti * 256 + (int)rank * PC::BM, brow = tj * BN + (int)rank * (BN / 2);
        int kb_lo;
        const int nkb = kblocks(q, tj, &kb_lo);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            give_up();
            report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 21);
            ok = false;
            break;
          }
          const int k0 = (kb_lo + kb) * PC::BK;
          const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
          if (rank == 0) tc::mbar_expect_tx(&full[stage], 2 * bytes);   // both CTAs' loads
          if constexpr (kMN) {
            // features [row0, row0 + 128) of k rows [k0, k0 + BK) as two 64-feature
            // chunks; the bias feature's chunk from the ones map
            // (m[2]: both chunks in one box, for blocks of whole chunks without the
            // bias feature; m[0] per chunk, zero past d; m[1] the ones matrix)
            const int bias = g.prob[q].bias_col, full = g.prob[q].mn_full;
            auto load_mn = [&](uint8_t* dst, int row0) {
              if (row0 + 128 <= full && (bias < row0 || bias >= row0 + 128)) {
                tc::tma_load_3d_pair(dst, &m[2], fb, 0, k0, row0 / 64);
                return;
              }
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int f = row0 + 64 * c;
                if (f == bias)
                  tc::tma_load_2d_pair(dst + c * PC::MN_CHUNK, &m[1], fb, 0, k0);
                else
                  tc::tma_load_2d_pair(dst + c * PC::MN_CHUNK, &m[0], fb, f, k0);
              }
            };
            if (!aib) load_mn(a_ptr(stage, 0), arow);
            load_mn(b_ptr(stage, 0), brow);
          } else {
            if (!aib) tc::tma_load_2d_pair(a_ptr(stage, 0), &m[0], fb, k0, arow);
            tc::tma_load_2d_pair(b_ptr(stage, 0), &m[2], fb, k0, brow);
            if (!kBF16) {
              if (!aib) tc::tma_load_2d_pair(a_ptr(stage, 1), &m[1], fb, k0, arow);
              tc::tma_load_2d_pair(b_ptr(stage, 1), &m[3], fb, k0, brow);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // ------------------------------ MMA issuer
      constexpr uint32_t idesc = tc::make_idesc(kBF16 ? 1 : 2, 256, BN);
      constexpr uint32_t idesc_c = tc::make_idesc(1, 256, BN);   // bf16 corrections
      int stage = 0;
      uint32_t phase = 0;
      int gsub = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        int q, ti, tj;
        grouped_tile<1>(g, t, &q, &ti, &tj);
        const bool aib = a_in_b(q, ti, tj);
        const bool corr = !kBF16 && g.prob[q].corr != 0;
        int kb_lo;
        const int nkb = kblocks(q, tj, &kb_lo);
        const int nsub = (nkb + kb_per_sub - 1) / kb_per_sub;
        for (int sub = 0; sub < nsub && ok; ++sub, ++gsub) {
          const int buf = gsub % PC::ACC, use = gsub / PC::ACC;
          if (!tc::mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag)) {
            report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 22);
            give_up();
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * BN);
          const int kb0 = sub * kb_per_sub, kb1 = min(nkb, kb0 + kb_per_sub);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::mbar_wait(&full[stage], phase, abort_flag)) {
              report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 23);
              give_up();
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const int lo1 = kBF16 ? 0 : 1;
            const uint32_t a_hi = tc::smem_u32(aib ? b_ptr(stage, 0) : a_ptr(stage, 0));
            const uint32_t b_hi = tc::smem_u32(b_ptr(stage, 0));
            const uint32_t a_lo = tc::smem_u32(aib ? b_ptr(stage, lo1) : a_ptr(stage, lo1));
            const uint32_t b_lo = tc::smem_u32(b_ptr(stage, lo1));
#pragma unroll
            for (int kk = 0; kk < PC::BK / PC::KMMA; ++kk) {
              const uint32_t off = kk * 32;
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              if (kMN) {   // 16 k = two 8-row groups further down both operands
                tc::umma_f16_pair(d, tc::sdesc_mnmajor_sw128(a_hi + kk * 2048, PC::MN_CHUNK),
                                  tc::sdesc_mnmajor_sw128(b_hi + kk * 2048, PC::MN_CHUNK),
                                  idesc | tc::kIdescMnA | tc::kIdescMnB, acc);
              } else if (kBF16) {
                tc::umma_f16_pair(d, tc::sdesc_kmajor_sw128(a_hi + off),
                                  tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
              } else if (corr) {
                tc::umma_tf32_pair(d, tc::sdesc_kmajor_sw128(a_hi + off),
                                   tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
                tc::umma_f16_pair(d, tc::sdesc_kmajor_sw128(a_lo + off),
                                  tc::sdesc_kmajor_sw128(b_lo + off), idesc_c, 1u);
              } else {
                tc::umma_tf32_pair(d, tc::sdesc_kmajor_sw128(a_hi + off),
                                   tc::sdesc_kmajor_sw128(b_hi + off), idesc, acc);
                tc::umma_tf32_pair(d, tc::sdesc_kmajor_sw128(a_hi + off),
                                   tc::sdesc_kmajor_sw128(b_lo + off), idesc, 1u);
                tc::umma_tf32_pair(d, tc::sdesc_kmajor_sw128(a_lo + off),
                                   tc::sdesc_kmajor_sw128(b_hi + off), idesc, 1u);
              }
            }
            tc::umma_commit_pair(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (ok) tc::umma_commit_pair(&acc_full[buf]);
        }
      }
    }
  } else {  // ------------------------------------------------ drain + epilogue
    const int qd = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;           // column block: [CW h, CW h + CW)
    const int row = 32 * qd + lane;
    float* xb = xbuf + (warp - 2) * 32 * PC::XP;
    const uint32_t acc_empty0 = tc::mapa(acc_empty, 0);
    int gsub = 0;
    bool ok = true;
    for (int t = pair; t < total && ok; t += npairs) {
      int q, ti, tj;
      grouped_tile<1>(g, t, &q, &ti, &tj);
      const TcEpilogue E = g.prob[q].e;   // by value (see gemm_body)
      const int64_t pM = g.prob[q].M, pN = g.prob[q].N;
      const int64_t r0 = (int64_t)ti * 256 + rank * PC::BM, c0 = (int64_t)tj * BN + h * CW;
      const int64_t gr = r0 + row;
      int kb_lo;
      const int nkb = kblocks(q, tj, &kb_lo);
      const int nsub = (nkb + kb_per_sub - 1) / kb_per_sub;
      auto prefetch_epilogue = [&]() {   // the tile's epilogue inputs into L2
        if (gr >= pM) return;
        if (EPI == TC_EPI_PRECOND && E.pw && gr < E.d_in) {
          for (int c = 0; c < CW; ++c) {
            const int64_t i = c0 + c;
            if (i >= pN) break;
            tc::prefetch_l2(E.pw + i * E.d_in + gr);
            tc::prefetch_l2(E.mw + i * E.d_in + gr);
          }
        }
      };
      const int pf_sub = max(0, nsub - 2);   // late enough that the lines stay in L2
      float sum[CW];
      float oscale;
      const float kin = sum_init<EPI, CW>(E, sum, c0, gr, pM, pN, &oscale);
      for (int sub = 0; sub < nsub; ++sub, ++gsub) {
        if (sub == pf_sub) prefetch_epilogue();
        const int buf = gsub % PC::ACC, use = gsub / PC::ACC;
        if (!tc::mbar_wait(&acc_full[buf], use & 1, abort_flag)) {
          report_error(g.prob[q].status, KFAC_ERR_TIMEOUT, g.prob[q].layer, 24);
          give_up();
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < CW / 16; ++cc) {
          float v[16];
          tc::tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * BN + h * CW + cc * 16),
                        v);
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[cc * 16 + i] = fmaf(kin, v[i], sum[cc * 16 + i]);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(acc_empty0 + (uint32_t)(buf * sizeof(uint64_t)));
      }
      if (!ok) break;
      epilogue_from_registers<EPI, CW, PC::XW, 8>(E, sum, xb, lane, qd, r0, c0, gr, pM, pN, oscale);
    }
  }
  tc::tc_fence_before();
  __syncwarp();
  tc::cluster_sync();   // every MMA of the pair has completed; no peer arrival is pending
  if (warp == 1) tc::tmem_dealloc_pair(tmem, PC::TMEM_COLS);
}

template <bool kBF16, int EPI, bool kMN>
__global__ void __maxnreg__(96) gemm_tc_pair_kernel(const __grid_constant__ GroupedTc g) {
  pair_body<kBF16, EPI, kMN>(g);
}

// ------------------------------------------------------------ wait self-test
// One thread waits, through the same bounded wait as the GEMM pipeline's
// roles, for an mbarrier phase that nothing completes: after `limit` clocks the
// wait gives up, the kernel records KFAC_ERR_TIMEOUT and returns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(DevStatus* st, long long limit) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &abort_flag, limit))
    report_error(st, KFAC_ERR_TIMEOUT, -1, 1);
}

// ------------------------------------------------------------------- pack
// X[c][r] = x-hat[r][c] for c < n, r < M; fp32 -> (hi, lo) TF32 halves; bf16 -> copy.
// One CTA moves a tile of kPackRows rows x 32 columns through shared memory
// (row pitch 33: conflict-free both ways): loads run along columns (coalesced
// rows of x-hat), stores along rows (coalesced rows of X); each thread keeps
// kPackRows / 8 loads in flight.
constexpr int kPackRows = 128;
template <typename T, bool kSplit>
__device__ __forceinline__ void pack_tile(const T* __restrict__ x, int64_t ld, int64_t M, int d,
                                          int n, int64_t Kp, void* out_hi, void* out_lo,
                                          int64_t r0, int c0) {
  __shared__ float tile[kPackRows][33];
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;  // 32 x 8
  float v[kPackRows / 8];
#pragma unroll
  for (int u = 0; u < kPackRows / 8; ++u) {
    const int64_t r = r0 + ty + 8 * u;
    const int c = c0 + tx;
    v[u] = 0.f;
    if (r < M && c < n) v[u] = c < d ? to_f32<T>(x[r * ld + c]) : 1.f;
  }
#pragma unroll
  for (int u = 0; u < kPackRows / 8; ++u) tile[ty + 8 * u][tx] = v[u];
  __syncthreads();
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {          // warp ty writes columns ty, ty + 8, ...
    const int c = c0 + ty + 8 * cc;
    if (c >= n) continue;
#pragma unroll
    for (int rr = 0; rr < kPackRows / 32; ++rr) {
      const int64_t r = r0 + 32 * rr + tx;
      if (r >= Kp) continue;
      const float w = tile[32 * rr + tx][ty + 8 * cc];
      if (kSplit) {
        const float hi = tc::to_tf32(w);
        static_cast<float*>(out_hi)[(int64_t)c * Kp + r] = hi;
        static_cast<float*>(out_lo)[(int64_t)c * Kp + r] = tc::to_tf32(w - hi);
      } else {
        static_cast<__nv_bfloat16*>(out_hi)[(int64_t)c * Kp + r] = __float2bfloat16_rn(w);
      }
    }
  }
}

// Gathered pack: X[c][r] for rows r of the input patches of a 2-D convolution
// over the NCHW tensor x (column c = (channel, kernel row, kernel column), zero
// outside the image; c = d is the ones column), or of an NCHW output gradient
// (1x1, unit stride).  Consecutive rows are consecutive output positions, which
// at unit stride are consecutive addresses of x, so loads and stores both run
// along rows and no transpose is needed: thread t takes row r0 + t % kPackRows
// and 16 of the tile's 32 columns, 16 loads in flight.  Each column's offset
// into an image and its kernel displacement come from a table the CTA builds
// once, so the per-element work is two bounds checks and an add.
template <typename T, bool kSplit>
__device__ __forceinline__ void pack_tile_conv(const T* __restrict__ x, const ConvSrc& g, int d,
                                               int n, int64_t M, int64_t Kp, void* out_hi,
                                               void* out_lo, int64_t r0, int c0) {
  __shared__ int64_t col_off[32];
  __shared__ int col_dy[32], col_dx[32];
  if (threadIdx.x < 32) {
    const int c = c0 + threadIdx.x;
    int64_t off = -1;
    int dy = 0, dx = 0;
    if (c < d) {
      const int khw = g.kh * g.kw, ci = c / khw, t = c - ci * khw, i = t / g.kw, j = t - i * g.kw;
      dy = i * g.dh;
      dx = j * g.dw;
      off = (int64_t)ci * g.H * g.W + (int64_t)dy * g.W + dx;
    }
    col_off[threadIdx.x] = off;   // -1: ones column or past n
    col_dy[threadIdx.x] = dy;
    col_dx[threadIdx.x] = dx;
  }
  __syncthreads();
  const int tr = threadIdx.x % kPackRows, half = threadIdx.x / kPackRows;
  const int64_t r = r0 + tr;
  const bool live = r < M;
  int64_t base = 0;
  int oy = 0, ox = 0;
  if (live) {
    const int64_t hw = (int64_t)g.Ho * g.Wo, img = r / hw;
    const int p = (int)(r - img * hw), oh = p / g.Wo, ow = p - oh * g.Wo;
    oy = oh * g.sh - g.ph;
    ox = ow * g.sw - g.pw;
    base = img * (int64_t)g.C * g.H * g.W + (int64_t)oy * g.W + ox;
  }
  float v[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int k = half * 16 + u, c = c0 + k;
    float val = 0.f;
    if (live && c < n) {
      const int64_t off = col_off[k];
      if (off < 0) {
        val = 1.f;   // c == d: the ones column
      } else {
        const int y = oy + col_dy[k], xx = ox + col_dx[k];
        if ((unsigned)y < (unsigned)g.H && (unsigned)xx < (unsigned)g.W)
          val = to_f32<T>(x[base + off]);
      }
    }
    v[u] = val;
  }
  if (r >= Kp) return;
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int c = c0 + half * 16 + u;
    if (c >= n) break;
    if (kSplit) {
      const float hi = tc::to_tf32(v[u]);
      static_cast<float*>(out_hi)[(int64_t)c * Kp + r] = hi;
      static_cast<float*>(out_lo)[(int64_t)c * Kp + r] = tc::to_tf32(v[u] - hi);
    } else {
      static_cast<__nv_bfloat16*>(out_hi)[(int64_t)c * Kp + r] = __float2bfloat16_rn(v[u]);
    }
  }
}

// Job q owns blocks [block_start[q], block_start[q+1]): its kPackRows x 32 tiles,
// row tiles fastest (a grid sized by the largest job in each dimension would
// schedule mostly empty blocks when the jobs differ in size).
struct PackGroup {
  PackJob job[kMaxPackJobs];
  int64_t block_start[kMaxPackJobs + 1];
  int count;
};

// bf16 pack of a row-major x-hat with 4-byte aligned column pairs (even ld, 4-byte
// aligned base): a CTA moves a 64-row x 64-column tile.  Each thread loads
// column pairs (c, c + 1) of two rows as 32-bit words, turns each 2 x 2 block
// around with byte permutes, and the words go through shared memory (pitch 33,
// conflict-free both ways) so that the stores, too, are 32-bit words along rows
// of X (128 contiguous bytes per warp).
constexpr int kPackBf2 = 64;
__device__ __forceinline__ uint32_t bf16_bits_at(const __nv_bfloat16* x, int64_t off, int c,
                                                 int d, int n) {
  if (c < d) return (uint32_t)__bfloat16_as_ushort(x[off + c]);
  return c == d && c < n ? 0x3F80u : 0u;   // the ones column (1.0), then nothing
}
__device__ __forceinline__ void pack_tile_bf16x2(const __nv_bfloat16* __restrict__ x, int64_t ld,
                                                 int64_t M, int d, int n, int64_t Kp,
                                                 __nv_bfloat16* out, int64_t r0, int c0) {
  __shared__ uint32_t s0[32][33], s1[32][33];
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;   // 32 x 8
  const int c = c0 + 2 * tx;
  uint32_t w[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t r = r0 + 2 * (ty + 8 * u) + e;
      uint32_t v = 0u;
      if (r < M) {
        if (c + 1 < d)
          v = __ldg(reinterpret_cast<const unsigned int*>(x + r * ld + c));
        else
          v = bf16_bits_at(x, r * ld, c, d, n) | (bf16_bits_at(x, r * ld, c + 1, d, n) << 16);
      }
      w[2 * u + e] = v;
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int br = ty + 8 * u;
    s0[tx][br] = __byte_perm(w[2 * u], w[2 * u + 1], 0x5410);   // column c, rows 2br, 2br+1
    s1[tx][br] = __byte_perm(w[2 * u], w[2 * u + 1], 0x7632);   // column c + 1
  }
  __syncthreads();
  const int64_t rr = r0 + 2 * tx;
  if (rr >= Kp) return;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int bc = ty + 8 * u;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int cc = c0 + 2 * bc + e;
      if (cc >= n) continue;
      *reinterpret_cast<uint32_t*>(out + (int64_t)cc * Kp + rr) = e ? s1[bc][tx] : s0[bc][tx];
    }
  }
}

__global__ void __launch_bounds__(256) pack_grouped_bf16x2_kernel(const __grid_constant__ PackGroup g) {
  pdl_wait();
  pdl_trigger();
  const int64_t b = blockIdx.x;
  int q = 0;
  while (q + 1 < g.count && b >= g.block_start[q + 1]) ++q;
  const PackJob& J = g.job[q];
  const int64_t Kp = J.Kp, local = b - g.block_start[q], rt = (Kp + kPackBf2 - 1) / kPackBf2;
  pack_tile_bf16x2(static_cast<const __nv_bfloat16*>(J.x), J.ld, J.M, J.d, J.n, Kp,
                   static_cast<__nv_bfloat16*>(J.hi), (local % rt) * kPackBf2,
                   (int)(local / rt) * kPackBf2);
}


// One kernel per source kind (kConv: every job of the launch is a gathered one),
// so the row-major pack keeps its small register footprint and occupancy.
template <typename T, bool kSplit, bool kConv>
__global__ void __launch_bounds__(256) pack_grouped_kernel(const __grid_constant__ PackGroup g) {
  pdl_wait();
  pdl_trigger();
  const int64_t b = blockIdx.x;
  int q = 0;
  while (q + 1 < g.count && b >= g.block_start[q + 1]) ++q;
  const PackJob& J = g.job[q];
  const int64_t Kp = J.Kp, local = b - g.block_start[q], rt = (Kp + kPackRows - 1) / kPackRows;
  if (kConv) {
    const ConvSrc cs = J.cs;
    pack_tile_conv<T, kSplit>(static_cast<const T*>(J.x), cs, J.d, J.n, J.M, Kp, J.hi, J.lo,
                              (local % rt) * kPackRows, (int)(local / rt) * 32);
  } else {
    pack_tile<T, kSplit>(static_cast<const T*>(J.x), J.ld, J.M, J.d, J.n, Kp, J.hi, J.lo,
                         (local % rt) * kPackRows, (int)(local / rt) * 32);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows x cols] row-major matrix (cols contiguous, pitch in elements), box of
// box_rows rows x 128 bytes, 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* m, const void* base, bool bf16, int64_t rows, int64_t cols,
              int64_t pitch, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int elt = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch * elt)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elt), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [rows x 64 chunks] (pitch in elements) seen as [chunks][rows][64]: a box
// of 2 chunks x box_rows rows x 64 elements lands in shared memory as two MN-major
// chunk tiles (128-byte swizzle), the layout two 2-D boxes of make_map would give.
bool make_chunk_map(CUtensorMap* m, const void* base, int64_t rows, int64_t chunks,
                    int64_t pitch, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)chunks};
  cuuint64_t strides[2] = {(cuuint64_t)(pitch * 2), 128u};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 2u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kBF16, int BN, int EPI>
bool set_smem_attr() {
  static bool done = false;
  static bool ok = false;
  if (!done) {
    ok = cudaFuncSetAttribute(gemm_tc_kernel<kBF16, BN, EPI>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)TcCfg<kBF16, BN>::SMEM) == cudaSuccess;
    done = true;
  }
  return ok;
}

// k elements per TMEM drain.  The tensor-core accumulator loses about half an ulp per
// accumulation (measured: ~6e-5 relative after 1024 bf16 MMAs into one accumulator),
// so no accumulator runs longer than 16 (bf16) or 16 x 3 (3xTF32) MMAs before its
// partial sum moves to fp32 registers.
constexpr int kKsubTf32 = 128;
constexpr int kKsubBf16 = 256;
// k elements per TMEM drain of the 256-wide persistent and CTA-pair bf16 products:
// 128 MMAs.  Measured on a 16384-row SYRK of o = 8192 against float64: 3.4e-7
// relative at 512, 7.1e-7 at 1024, 1.9e-6 at 2048, 2.4e-5 with no drain (the
// factor gate is 1e-5).  Each drain costs the drain warps about 2000 cycles and
// the pair's two accumulators let the MMA run only two drain periods ahead of a
// tile's epilogue: the transformer factor phase takes 7.65 ms at 1024 and
// 7.34 ms at 2048.
constexpr int kKsubBf16Wide = 2048;
// Products with a wave of wide tiles run on CTA pairs (256 x 256 tiles).
constexpr bool kWidePairs = true;

template <bool kBF16, int BN, int EPI>
kfac_status launch_kernel(unsigned grid, const CUtensorMap& ah, const CUtensorMap& al,
                          const CUtensorMap& bh, const CUtensorMap& bl, const GemmTcParams& p,
                          cudaStream_t st) {
  if (!set_smem_attr<kBF16, BN, EPI>()) return KFAC_ERR_CUDA;
  if (p.csize > 1 || p.mc) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TcCfg<kBF16, BN>::THREADS);
    cfg.dynamicSmemBytes = TcCfg<kBF16, BN>::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.mc ? 2u : (unsigned)p.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel<kBF16, BN, EPI>, ah, al, bh, bl, p) != cudaSuccess)
      return KFAC_ERR_CUDA;
  } else {
    launch_pdl(gemm_tc_kernel<kBF16, BN, EPI>, dim3(grid), dim3(TcCfg<kBF16, BN>::THREADS),
               TcCfg<kBF16, BN>::SMEM, st, ah, al, bh, bl, p);
  }
  count_launch();
  return check_launch();
}

}  // namespace

int64_t tc_pitch(int64_t cols, bool bf16) { return cdiv(cols, bf16 ? 8 : 4) * (bf16 ? 8 : 4); }

kfac_status launch_wait_selftest(kfac_ctx* h, int64_t wait_cycles, cudaStream_t st) {
  launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, st, h->status(), (long long)wait_cycles);
  count_launch();
  return check_launch();
}

kfac_status launch_pack_grouped(const PackJob* jobs, int count, bool bf16, cudaStream_t st) {
  PackGroup g;
  for (int conv = 0; conv < 2; ++conv) {   // row-major jobs, then gathered ones
    std::vector<const PackJob*> sel;
    for (int q = 0; q < count; ++q)
      if ((jobs[q].conv != 0) == (conv != 0)) sel.push_back(&jobs[q]);
    for (size_t c0 = 0; c0 < sel.size(); c0 += kMaxPackJobs) {
      std::memset(&g, 0, sizeof(g));
      const int cnt = (int)std::min<size_t>(kMaxPackJobs, sel.size() - c0);
      // bf16 row-major sources whose column pairs are 4-byte aligned take the paired pack
      bool pairs = bf16 && !conv;
      for (int q = 0; q < cnt && pairs; ++q)
        pairs = sel[c0 + q]->ld % 2 == 0 && (uintptr_t)sel[c0 + q]->x % 4 == 0;
      int64_t blocks = 0;
      for (int q = 0; q < cnt; ++q) {
        g.job[q] = *sel[c0 + q];
        g.block_start[q] = blocks;
        blocks += pairs ? cdiv(g.job[q].Kp, kPackBf2) * cdiv(g.job[q].n, kPackBf2)
                        : cdiv(g.job[q].Kp, kPackRows) * cdiv(g.job[q].n, 32);
      }
      g.block_start[cnt] = blocks;
      g.count = cnt;
      const dim3 grid((unsigned)blocks);
      if (pairs) {
        launch_pdl(pack_grouped_bf16x2_kernel, grid, dim3(256), 0, st, g);
      } else if (bf16) {
        if (conv)
          launch_pdl(pack_grouped_kernel<__nv_bfloat16, false, true>, grid, dim3(256), 0, st, g);
        else
          launch_pdl(pack_grouped_kernel<__nv_bfloat16, false, false>, grid, dim3(256), 0, st, g);
      } else {
        if (conv)
          launch_pdl(pack_grouped_kernel<float, true, true>, grid, dim3(256), 0, st, g);
        else
          launch_pdl(pack_grouped_kernel<float, true, false>, grid, dim3(256), 0, st, g);
      }
      count_launch();
      if (kfac_status e = check_launch()) return e;
    }
  }
  return KFAC_OK;
}

size_t tc_pack_bytes(int n, int64_t max_rows, bool bf16) {
  const int64_t Kp = tc_pitch(max_rows, bf16);
  return (size_t)n * Kp * (bf16 ? 2 : 8);
}

size_t tc_part_floats() { return (size_t)num_sms() * 128 * 256; }

// Split-K shape for `s` wanted splits of a reduction of length K: clusters of
// csize = min(8, s) splits (the portable cluster size) times `groups` cluster
// partials, each split a whole number of ksub steps.  `max_groups` bounds the
// cluster partials the scratch can hold.
struct SplitShape {
  int splits, csize;
  int64_t kps;
};
SplitShape split_shape(int64_t s, int64_t K, int unit, int64_t max_groups, int csize_fixed = 0) {
  SplitShape r;
  s = std::max<int64_t>(1, std::min<int64_t>(s, std::max<int64_t>(1, K / 256)));
  r.csize = csize_fixed > 0 ? csize_fixed : (int)std::min<int64_t>(8, s);
  int64_t g = cdiv(s, r.csize);
  g = std::max<int64_t>(1, std::min<int64_t>(g, max_groups));
  r.splits = (int)(r.csize * g);
  r.kps = cdiv(cdiv(K, r.splits), unit) * unit;
  return r;
}

template <int BN>
kfac_status dispatch(bool bf16, int epi, unsigned grid, const CUtensorMap& ah,
                     const CUtensorMap& al, const CUtensorMap& bh, const CUtensorMap& bl,
                     const GemmTcParams& p, cudaStream_t st) {
  if (epi == TC_EPI_SYRK)
    return bf16 ? launch_kernel<true, BN, TC_EPI_SYRK>(grid, ah, al, bh, bl, p, st)
                : launch_kernel<false, BN, TC_EPI_SYRK>(grid, ah, al, bh, bl, p, st);
  if (epi == TC_EPI_SPLIT)
    return bf16 ? launch_kernel<true, BN, TC_EPI_SPLIT>(grid, ah, al, bh, bl, p, st)
                : launch_kernel<false, BN, TC_EPI_SPLIT>(grid, ah, al, bh, bl, p, st);
  return bf16 ? launch_kernel<true, BN, TC_EPI_PRECOND>(grid, ah, al, bh, bl, p, st)
              : launch_kernel<false, BN, TC_EPI_PRECOND>(grid, ah, al, bh, bl, p, st);
}

kfac_status launch_wide_persistent(kfac_ctx* h, bool bf16, int epi, const TcProblem* probs,
                                   int count, cudaStream_t st, bool pair);

// the correction form pairs an A form with a B form: both operands or neither,
// fp32 operands in distinct arrays
bool corr_ok(bool bf16, const TcOperand& A, const TcOperand& B, bool same_ab) {
  return A.corr == B.corr && (!A.corr || (!bf16 && !same_ab));
}

kfac_status launch_gemm_tc(kfac_ctx* h, int layer, bool bf16, int epi, const TcOperand& A,
                           const TcOperand& B, bool same_ab, bool upper, int64_t M, int64_t N,
                           int64_t K, const TcEpilogue& e, cudaStream_t st, int kmode) {
  constexpr int BM = 128;
  const int sms = num_sms();
  if (!corr_ok(bf16, A, B, same_ab)) return KFAC_ERR_INVALID_ARG;
  // Tile width: 128 x 256 halves the shared-memory traffic per MMA flop of
  // 128 x 128, which pays on long reductions or when there are tiles enough to
  // fill the GPU; short, small products keep 128 x 128 for parallelism.
  auto count = [&](int bn) {
    const int tm = (int)cdiv(M, BM), tn = (int)cdiv(N, bn);
    return upper ? upper_tile_count(tm, tn, bn / BM) : (int64_t)tm * tn;
  };
  if (count(256) >= sms) {   // a wave of wide tiles at least: the persistent kernel
    TcProblem pr{};
    pr.A = A;
    pr.B = B;
    pr.same_ab = same_ab;
    pr.upper = upper;
    pr.M = M;
    pr.N = N;
    pr.K = K;
    pr.e = e;
    pr.layer = layer;
    pr.kmode = kmode;
    return launch_wide_persistent(h, bf16, epi, &pr, 1, st, kWidePairs);
  }
  const int BN = ((bf16 && K >= 8192) || count(256) >= sms) ? 256 : 128;
  // With at least a wave of tiles and no split-K, neighbouring tiles of one
  // column run as a cluster pair that loads the shared B tile once: each CTA
  // fetches half of its rows and multicasts them to both.
  const bool mc = count(BN) >= sms;
  const int b_box = mc ? BN / 2 : BN;
  CUtensorMap ah, al, bh, bl;
  if (!make_map(&ah, A.hi, bf16, A.rows, K, A.pitch, BM)) return KFAC_ERR_CUDA;
  if (!make_map(&bh, B.hi, bf16, B.rows, K, B.pitch, b_box)) return KFAC_ERR_CUDA;
  if (bf16) {
    al = ah;
    bl = bh;
  } else {
    if (!make_map(&al, A.lo, false, A.rows, K, A.pitch, BM)) return KFAC_ERR_CUDA;
    if (!make_map(&bl, B.lo, false, B.rows, K, B.pitch, b_box)) return KFAC_ERR_CUDA;
  }
  GemmTcParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (int)cdiv(M, BM);
  p.tiles_n = (int)cdiv(N, BN);
  p.upper = upper ? 1 : 0;
  p.same_ab = same_ab ? 1 : 0;
  p.kmode = kmode;
  p.corr = A.corr;
  const int64_t tiles = count(BN);
  // enough CTAs for one wave when the output has fewer tiles than SMs
  const int unit = bf16 ? kKsubBf16 : kKsubTf32;
  const int64_t max_groups =
      std::max<int64_t>(1, std::min<int64_t>((int64_t)(h->part_floats / ((size_t)tiles * BM * BN)),
                                             (int64_t)(h->n_tickets / ((size_t)tiles * 8))));
  // Fewer tiles than SMs: the split count minimising wave-quantised time,
  // ceil(tiles s / SMs) x (1/s + c0), where c0 is a CTA's fixed cost (prologue,
  // epilogue, reduction: ~8 us measured) relative to the tile's whole main loop
  // at the tensor rate of one SM.
  int64_t want = 1;
  if (tiles < sms) {
    const double sm_rate = (bf16 ? 2.25e15 : 1.1e15 / 3.0) / sms;   // flop/s per SM
    const double t_tile = 2.0 * BM * BN * (double)K / sm_rate;          // seconds
    const double c0 = 8e-6 / t_tile;
    double best = 1.0 + c0;
    const int64_t smax = std::max<int64_t>(1, std::min<int64_t>(K / 256, 4 * sms));
    for (int64_t sp = 2; sp <= smax; ++sp) {
      const double cost = (double)cdiv(tiles * sp, sms) * (1.0 / (double)sp + c0);
      if (cost < best - 1e-12) {
        best = cost;
        want = sp;
      }
    }
  }
  const SplitShape sh = split_shape(want, K, unit, max_groups);
  p.splits = sh.splits;
  p.csize = sh.csize;
  p.k_per_split = sh.kps;
  p.ksub = unit;
  p.part = h->at<float>(epi == TC_EPI_SYRK ? h->off_part : h->off_part_k4);
  p.tickets = h->at<int>(epi == TC_EPI_SYRK ? h->off_tickets : h->off_tickets_k4);
  p.status = h->status();
  p.layer = layer;
  p.e = e;
  unsigned grid = (unsigned)(tiles * p.splits);
  if (mc) {   // tiles >= SMs: split_shape gave one split
    p.mc = 1;
    grid = (unsigned)mc_tile_count(p.tiles_m, p.tiles_n, BN / BM, upper);
  }
  return BN == 256 ? dispatch<256>(bf16, epi, grid, ah, al, bh, bl, p, st)
                   : dispatch<128>(bf16, epi, grid, ah, al, bh, bl, p, st);
}

template <bool kBF16, int EPI, int BN>
kfac_status launch_persistent_kernel(const GroupedTc& g, cudaStream_t st) {
  using PC = PersistCfg<kBF16, BN>;
  static bool attr_ok = cudaFuncSetAttribute(PersistKernel<kBF16, EPI, BN>::fn,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)PC::SMEM) == cudaSuccess;
  if (!attr_ok) {
    check_launch();   // records the attribute error, if it is still pending
    return KFAC_ERR_CUDA;
  }
  const int total = g.block_start[g.count];
  const unsigned grid = (unsigned)std::min<int>(total, num_sms());
  launch_pdl(PersistKernel<kBF16, EPI, BN>::fn, dim3(grid), dim3(PC::THREADS), PC::SMEM, st, g);
  count_launch();
  return check_launch();
}


template <bool kBF16, int EPI, bool kMN = false>
kfac_status launch_pair_kernel(const GroupedTc& g, cudaStream_t st) {
  using PC = PairCfg<kBF16, kMN>;
  static bool attr_ok = cudaFuncSetAttribute(gemm_tc_pair_kernel<kBF16, EPI, kMN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)PC::SMEM) == cudaSuccess;
  if (!attr_ok) {
    check_launch();
    return KFAC_ERR_CUDA;
  }
  const int total = g.block_start[g.count];
  const int pairs = std::max(1, std::min<int>(total, num_sms() / 2));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3(PC::THREADS);
  cfg.dynamicSmemBytes = PC::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<kBF16, EPI, kMN>, g);
  count_launch();
  return check_launch();
}

// Products that fill at least a wave of 128 x 256 tiles by themselves, no
// split-K: persistent launches of up to kMaxGroup of them, each tile's epilogue
// overlapped with the next tile's main loop.  256 x 256 tiles on CTA pairs
// (pair), or 128 x 256 tiles on single CTAs.
kfac_status launch_wide_persistent(kfac_ctx* h, bool bf16, int epi, const TcProblem* probs,
                                   int count, cudaStream_t st, bool pair) {
  constexpr int BN = 256;
  const int BM = pair ? 256 : 128;                   // rows of a tile
  const int box_a = 128, box_b = pair ? 128 : BN;    // rows of A and B each CTA loads
  // Longest reductions first: a launch hands its tiles to the CTAs round-robin in
  // problem order, so its last, partly filled round then holds the shortest tiles
  // (the transformer set's preconditioning: 10.30 -> 9.93-10.02 ms).
  std::vector<TcProblem> by_k(probs, probs + count);
  std::stable_sort(by_k.begin(), by_k.end(),
                   [](const TcProblem& a, const TcProblem& b) { return a.K > b.K; });
  probs = by_k.data();
  std::unique_ptr<GroupedTc> g(new GroupedTc());
  for (int c0 = 0; c0 < count; c0 += kMaxGroup) {
    std::memset(g.get(), 0, sizeof(GroupedTc));
    const int cnt = std::min(kMaxGroup, count - c0);
    // one drain period for the launch (the kernel reads it from its first problem)
    const int unit = bf16 ? kKsubBf16Wide : probs[c0].drain_k > 0 ? probs[c0].drain_k : kKsubTf32;
    int blocks = 0;
    for (int i = 0; i < cnt; ++i) {
      const TcProblem& pr = probs[c0 + i];
      CUtensorMap* m = &g->maps[4 * i];
      if (!make_map(&m[0], pr.A.hi, bf16, pr.A.rows, pr.K, pr.A.pitch, box_a)) return KFAC_ERR_CUDA;
      if (!make_map(&m[2], pr.B.hi, bf16, pr.B.rows, pr.K, pr.B.pitch, box_b)) return KFAC_ERR_CUDA;
      GemmTcParams& pp = g->prob[i];
      if (bf16) {
        m[1] = m[0];
        m[3] = m[2];
      } else {
        if (!make_map(&m[1], pr.A.lo, false, pr.A.rows, pr.K, pr.A.pitch, box_a))
          return KFAC_ERR_CUDA;
        if (!make_map(&m[3], pr.B.lo, false, pr.B.rows, pr.K, pr.B.pitch, box_b))
          return KFAC_ERR_CUDA;
      }
      pp.M = pr.M;
      pp.N = pr.N;
      pp.K = pr.K;
      pp.tiles_m = (int)cdiv(pr.M, BM);
      pp.tiles_n = (int)cdiv(pr.N, BN);
      pp.upper = pr.upper ? 1 : 0;
      pp.same_ab = pr.same_ab ? 1 : 0;
      pp.kmode = pr.kmode;
      pp.colmajor = pr.M < pr.N ? 1 : 0;
      pp.corr = pr.A.corr;
      pp.splits = 1;
      pp.csize = 1;
      pp.k_per_split = cdiv(pr.K, unit) * unit;
      pp.ksub = unit;
      pp.status = h->status();
      pp.layer = pr.layer;
      pp.e = pr.e;
      g->block_start[i] = blocks;
      blocks += (int)(pr.upper ? upper_tile_count(pp.tiles_m, pp.tiles_n, BN / BM)
                               : (int64_t)pp.tiles_m * pp.tiles_n);
    }
    g->block_start[cnt] = blocks;
    g->count = cnt;
    g->csize = 1;
    kfac_status e;
    if (pair) {
      if (epi == TC_EPI_SYRK)
        e = bf16 ? launch_pair_kernel<true, TC_EPI_SYRK>(*g, st)
                 : launch_pair_kernel<false, TC_EPI_SYRK>(*g, st);
      else if (epi == TC_EPI_SPLIT)
        e = bf16 ? launch_pair_kernel<true, TC_EPI_SPLIT>(*g, st)
                 : launch_pair_kernel<false, TC_EPI_SPLIT>(*g, st);
      else
        e = bf16 ? launch_pair_kernel<true, TC_EPI_PRECOND>(*g, st)
                 : launch_pair_kernel<false, TC_EPI_PRECOND>(*g, st);
    } else if (epi == TC_EPI_SYRK) {
      e = bf16 ? launch_persistent_kernel<true, TC_EPI_SYRK, BN>(*g, st)
               : launch_persistent_kernel<false, TC_EPI_SYRK, BN>(*g, st);
    } else if (epi == TC_EPI_SPLIT) {
      e = bf16 ? launch_persistent_kernel<true, TC_EPI_SPLIT, BN>(*g, st)
               : launch_persistent_kernel<false, TC_EPI_SPLIT, BN>(*g, st);
    } else {
      e = bf16 ? launch_persistent_kernel<true, TC_EPI_PRECOND, BN>(*g, st)
               : launch_persistent_kernel<false, TC_EPI_PRECOND, BN>(*g, st);
    }
    if (e) return e;
  }
  return KFAC_OK;
}

int64_t syrk_pair_tiles(int n) {
  const int t = (int)cdiv(n, 256);
  return (int64_t)t * (t + 1) / 2;
}

bool syrk_direct_layout_ok(const kfac_ctx* h, const void* x, int64_t ld, int64_t rows, int d,
                           int has_bias) {
  if (ld % 8 != 0 || reinterpret_cast<uintptr_t>(x) % 16 != 0 || rows < 1) return false;
  if (has_bias && (d % 64 != 0 || h->ones_rows < rows)) return false;
  return true;
}

// The factor SYRKs of bf16 layers read straight from the callers' activations:
// a [K x d] row-major array is, for C = X^T X, an MN-major operand (features
// contiguous), which the bf16 MMA takes through its transpose bits.  A 3-D tensor
// map over x loads 128 features x 128 k per box (2-D maps, 64 features per box,
// for blocks with the bias feature or a ragged edge); the ones column of x-hat
// (feature d of a layer with a bias) loads from a [K x 64] matrix whose first
// column is one.
// Saves the pack's read and write of every input.  CTA pairs as in
// launch_wide_persistent; groups of kMaxGroup.
kfac_status launch_syrk_direct(kfac_ctx* h, const TcProblem* probs, int count, cudaStream_t st) {
  constexpr int BN = 256;
  std::unique_ptr<GroupedTc> g(new GroupedTc());
  for (int c0 = 0; c0 < count; c0 += kMaxGroup) {
    std::memset(g.get(), 0, sizeof(GroupedTc));
    const int cnt = std::min(kMaxGroup, count - c0);
    int blocks = 0;
    for (int i = 0; i < cnt; ++i) {
      const TcProblem& pr = probs[c0 + i];
      CUtensorMap* m = &g->maps[4 * i];
      constexpr int kb = PairCfg<true, true>::BK;   // k rows per box
      if (!make_map(&m[0], pr.A.hi, true, pr.K, pr.A.rows, pr.A.pitch, kb)) return KFAC_ERR_CUDA;
      if (pr.bias_col >= 0) {
        if (!make_map(&m[1], h->ws + h->off_ones, true, pr.K, 64, 64, kb)) return KFAC_ERR_CUDA;
      } else {
        m[1] = m[0];
      }
      const int full = (int)(pr.A.rows / 64 * 64);
      if (full >= 64) {
        if (!make_chunk_map(&m[2], pr.A.hi, pr.K, pr.A.rows / 64, pr.A.pitch, kb)) return KFAC_ERR_CUDA;
      } else {
        m[2] = m[0];
      }
      m[3] = m[1];
      GemmTcParams& pp = g->prob[i];
      pp.M = pr.M;
      pp.N = pr.N;
      pp.K = pr.K;
      pp.tiles_m = pp.tiles_n = (int)cdiv(pr.M, BN);
      pp.upper = 1;
      pp.same_ab = 1;
      pp.splits = 1;
      pp.csize = 1;
      pp.k_per_split = cdiv(pr.K, kKsubBf16Wide) * kKsubBf16Wide;
      pp.ksub = kKsubBf16Wide;
      pp.bias_col = pr.bias_col;
      pp.mn_full = full;
      pp.status = h->status();
      pp.layer = pr.layer;
      pp.e = pr.e;
      g->block_start[i] = blocks;
      blocks += (int)syrk_pair_tiles((int)pr.M);
    }
    g->block_start[cnt] = blocks;
    g->count = cnt;
    g->csize = 1;
    if (kfac_status e = launch_pair_kernel<true, TC_EPI_SYRK, true>(*g, st)) return e;
  }
  return KFAC_OK;
}

template <bool kBF16, int EPI>
kfac_status launch_grouped_kernel(unsigned grid, const GroupedTc& g, cudaStream_t st) {
  if (g.csize == 1 && g.prob[0].splits == 1) return launch_persistent_kernel<kBF16, EPI, 128>(g, st);
  static bool attr_ok = cudaFuncSetAttribute(gemm_tc_grouped_kernel<kBF16, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)TcCfg<kBF16, 128>::SMEM) == cudaSuccess;
  if (!attr_ok) return KFAC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TcCfg<kBF16, 128>::THREADS);
  cfg.dynamicSmemBytes = TcCfg<kBF16, 128>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, gemm_tc_grouped_kernel<kBF16, EPI>, g) != cudaSuccess)
    return KFAC_ERR_CUDA;
  count_launch();
  return check_launch();
}

// Independent products of one epilogue kind in as few launches as possible
// (128 x 128 tiles, up to kMaxGroup products per launch).  Each product gets its
// own split-K count so that every CTA carries about the same share of the
// launch's k-steps; products that need no split and products that do go to
// separate launches (the cluster size is a launch attribute), and a launch is
// cut when the split-K scratch is full.
kfac_status launch_gemm_tc_grouped(kfac_ctx* h, bool bf16, int epi, const TcProblem* probs,
                                   int count, cudaStream_t st) {
  for (int q = 0; q < count; ++q)
    if (!corr_ok(bf16, probs[q].A, probs[q].B, probs[q].same_ab)) return KFAC_ERR_INVALID_ARG;
  if (count == 1) {
    const TcProblem& q = probs[0];
    return launch_gemm_tc(h, q.layer, bf16, epi, q.A, q.B, q.same_ab, q.upper, q.M, q.N, q.K,
                          q.e, st, q.kmode);
  }
  constexpr int BM = 128, BN = 128;
  constexpr size_t NT = (size_t)BM * BN;
  const int sms = num_sms();
  const int unit = bf16 ? kKsubBf16 : kKsubTf32;
  // Products that fill a wave of 128 x 256 tiles by themselves go to the wide
  // persistent launches; the rest share grouped launches.
  std::vector<TcProblem> small, wide_probs;
  for (int q = 0; q < count; ++q) {
    const TcProblem& pr = probs[q];
    const int tm = (int)cdiv(pr.M, BM), tn = (int)cdiv(pr.N, 256);
    const int64_t wide = pr.upper ? upper_tile_count(tm, tn, 2) : (int64_t)tm * tn;
    (wide >= sms ? wide_probs : small).push_back(pr);
  }
  if (!wide_probs.empty())
    if (kfac_status e = launch_wide_persistent(h, bf16, epi, wide_probs.data(),
                                               (int)wide_probs.size(), st, kWidePairs))
      return e;
  if (small.empty()) return KFAC_OK;
  if ((int)small.size() < count) return launch_gemm_tc_grouped(h, bf16, epi, small.data(), (int)small.size(), st);
  std::vector<int64_t> tiles(count), want(count);
  int64_t total_units = 0;
  for (int q = 0; q < count; ++q) {
    const TcProblem& pr = probs[q];
    const int tm = (int)cdiv(pr.M, BM), tn = (int)cdiv(pr.N, BN);
    tiles[q] = pr.upper ? upper_tile_count(tm, tn, 1) : (int64_t)tm * tn;
    total_units += tiles[q] * cdiv(pr.K, unit);
  }
  // k-steps per CTA if the whole group were spread over one wave
  const int64_t chunk = std::max<int64_t>(2, cdiv(total_units, sms));
  for (int q = 0; q < count; ++q)
    want[q] = std::max<int64_t>(1, cdiv(cdiv(probs[q].K, unit), chunk));
  // The products that need no split run on CTA pairs (256 x 256 tiles) when that
  // is faster after wave quantisation: a pair tile is four 128 x 128 tiles of work
  // on two SMs at about 0.75 of the single-CTA time per flop (measured: the pair's
  // MMA is fed twice the operand bytes per shared-memory byte).
  {
    std::vector<TcProblem> unsplit;
    double t1 = 0, t2 = 0, k1 = 0, k2 = 0;
    for (int q = 0; q < count; ++q) {
      if (want[q] != 1) continue;
      const TcProblem& pr = probs[q];
      const int tm = (int)cdiv(pr.M, 256), tn = (int)cdiv(pr.N, 256);
      const int64_t pt = pr.upper ? upper_tile_count(tm, tn, 1) : (int64_t)tm * tn;
      t1 += (double)tiles[q];
      k1 += (double)tiles[q] * (double)pr.K;
      t2 += (double)pt;
      k2 += (double)pt * (double)pr.K;
      unsplit.push_back(pr);
    }
    if (!unsplit.empty() && t2 >= sms / 2) {
      const double cost1 = std::ceil(t1 / sms) * (k1 / t1);
      const double cost2 = std::ceil(t2 / (sms / 2)) * 2.0 * 0.75 * (k2 / t2);
      if (cost2 < cost1) {
        if (kfac_status e = launch_wide_persistent(h, bf16, epi, unsplit.data(),
                                                   (int)unsplit.size(), st, true))
          return e;
        for (int q = 0; q < count; ++q)
          if (want[q] == 1) want[q] = 0;   // done
      }
    }
  }
  std::unique_ptr<GroupedTc> g(new GroupedTc());
  for (int pass = 0; pass < 2; ++pass) {   // pass 0: unsplit products; pass 1: split ones
    const int csize = pass == 0 ? 1 : 8;
    std::memset(g.get(), 0, sizeof(GroupedTc));
    g->csize = csize;
    int blocks = 0;
    size_t part_used = 0, tick_used = 0;
    auto flush = [&]() -> kfac_status {
      if (g->count == 0) return KFAC_OK;
      g->block_start[g->count] = blocks;
      kfac_status e;
      if (epi == TC_EPI_SYRK)
        e = bf16 ? launch_grouped_kernel<true, TC_EPI_SYRK>(blocks, *g, st)
                 : launch_grouped_kernel<false, TC_EPI_SYRK>(blocks, *g, st);
      else if (epi == TC_EPI_SPLIT)
        e = bf16 ? launch_grouped_kernel<true, TC_EPI_SPLIT>(blocks, *g, st)
                 : launch_grouped_kernel<false, TC_EPI_SPLIT>(blocks, *g, st);
      else
        e = bf16 ? launch_grouped_kernel<true, TC_EPI_PRECOND>(blocks, *g, st)
                 : launch_grouped_kernel<false, TC_EPI_PRECOND>(blocks, *g, st);
      std::memset(g.get(), 0, sizeof(GroupedTc));
      g->csize = csize;
      blocks = 0;
      part_used = tick_used = 0;
      return e;
    };
    for (int q = 0; q < count; ++q) {
      if (want[q] == 0 || (want[q] > 1) != (pass == 1)) continue;
      const TcProblem& pr = probs[q];
      SplitShape sh{1, 1, cdiv(pr.K, unit) * unit};
      if (pass == 1) {
        // cluster partials this product may use: what the scratch holds by itself
        const int64_t max_groups = std::max<int64_t>(
            1, std::min<int64_t>((int64_t)(h->part_floats / (tiles[q] * NT)),
                                 (int64_t)(h->n_tickets / (tiles[q] * csize))));
        sh = split_shape(want[q], pr.K, unit, max_groups, csize);
      }
      const int G = sh.splits / sh.csize;
      const size_t pneed = G > 1 ? (size_t)tiles[q] * G * NT : 0;
      const size_t tneed = G > 1 ? (size_t)tiles[q] * csize : 0;
      if (g->count == kMaxGroup || part_used + pneed > h->part_floats ||
          tick_used + tneed > h->n_tickets)
        if (kfac_status e = flush()) return e;
      const int i = g->count;
      CUtensorMap* m = &g->maps[4 * i];
      if (!make_map(&m[0], pr.A.hi, bf16, pr.A.rows, pr.K, pr.A.pitch, BM)) return KFAC_ERR_CUDA;
      if (!make_map(&m[2], pr.B.hi, bf16, pr.B.rows, pr.K, pr.B.pitch, BN)) return KFAC_ERR_CUDA;
      if (bf16) {
        m[1] = m[0];
        m[3] = m[2];
      } else {
        if (!make_map(&m[1], pr.A.lo, false, pr.A.rows, pr.K, pr.A.pitch, BM)) return KFAC_ERR_CUDA;
        if (!make_map(&m[3], pr.B.lo, false, pr.B.rows, pr.K, pr.B.pitch, BN)) return KFAC_ERR_CUDA;
      }
      GemmTcParams& pp = g->prob[i];
      pp.M = pr.M;
      pp.N = pr.N;
      pp.K = pr.K;
      pp.tiles_m = (int)cdiv(pr.M, BM);
      pp.tiles_n = (int)cdiv(pr.N, BN);
      pp.upper = pr.upper ? 1 : 0;
      pp.same_ab = pr.same_ab ? 1 : 0;
      pp.kmode = pr.kmode;
      pp.colmajor = pr.M < pr.N ? 1 : 0;
      pp.corr = pr.A.corr;
      pp.splits = sh.splits;
      pp.csize = sh.csize;
      pp.k_per_split = sh.kps;
      pp.ksub = unit;
      pp.part = h->at<float>(epi == TC_EPI_SYRK ? h->off_part : h->off_part_k4) + part_used;
      pp.tickets = h->at<int>(epi == TC_EPI_SYRK ? h->off_tickets : h->off_tickets_k4) + tick_used;
      pp.status = h->status();
      pp.layer = pr.layer;
      pp.e = pr.e;
      g->block_start[i] = blocks;
      blocks += (int)(tiles[q] * sh.splits);
      part_used += pneed;
      tick_used += tneed;
      ++g->count;
    }
    if (kfac_status e = flush()) return e;
  }
  return KFAC_OK;
}

// F <- beta F + alpha x-hat^T x-hat on the tensor cores (K1).
kfac_status launch_syrk_tc(kfac_ctx* h, int layer, const void* x, int64_t ld, int64_t rows, int d,
                           int n, int has_bias, bool bf16, float alpha, float beta, float* F,
                           cudaStream_t st) {
  if (bf16 && syrk_direct_layout_ok(h, x, ld, rows, d, has_bias) &&
      syrk_pair_tiles(n) >= num_sms() / 2) {   // in place, no pack (launch_syrk_direct)
    TcProblem q{};
    q.A = TcOperand{x, nullptr, d, ld};
    q.B = q.A;
    q.same_ab = true;
    q.upper = true;
    q.M = q.N = n;
    q.K = rows;
    q.bias_col = has_bias ? d : -1;
    q.e.alpha = alpha;
    q.e.beta = beta;
    q.e.C = F;
    q.e.ldc = n;
    q.layer = layer;
    return launch_syrk_direct(h, &q, 1, st);
  }
  const int64_t Kp = tc_pitch(rows, bf16);
  if ((size_t)n * Kp * (bf16 ? 2 : 8) > h->tcpack_bytes) return KFAC_ERR_WORKSPACE;
  void* hi = h->ws + h->off_tcpack;
  void* lo = bf16 ? nullptr : (void*)(h->ws + h->off_tcpack + (size_t)n * Kp * 4);
  {
    PackJob j{};
    j.x = x;
    j.ld = ld;
    j.M = rows;
    j.d = d;
    j.n = n;
    j.Kp = Kp;
    j.hi = hi;
    j.lo = lo;
    if (kfac_status e = launch_pack_grouped(&j, 1, bf16, st)) return e;
  }
  TcOperand X{hi, lo, n, Kp};
  TcEpilogue e{};
  e.alpha = alpha;
  e.beta = beta;
  e.C = F;
  e.ldc = n;
  return launch_gemm_tc(h, layer, bf16, TC_EPI_SYRK, X, X, true, true, n, n, rows, e, st);
}

kfac_status launch_syrk_tc_batched(kfac_ctx* h, const SyrkSpec* specs, int count,
                                   cudaStream_t st) {
  std::vector<PackJob> pj;
  std::vector<TcProblem> pr;
  size_t used = 0;
  auto flush = [&]() -> kfac_status {
    if (pr.empty()) return KFAC_OK;
    kfac_status e = launch_pack_grouped(pj.data(), (int)pj.size(), false, st);
    if (e == KFAC_OK) e = launch_gemm_tc_grouped(h, false, TC_EPI_SYRK, pr.data(), (int)pr.size(), st);
    pj.clear();
    pr.clear();
    used = 0;
    return e;
  };
  for (int i = 0; i < count; ++i) {
    const SyrkSpec& q = specs[i];
    const int64_t Kp = tc_pitch(q.rows, false);
    const size_t raw = (size_t)q.n * Kp * 8, bytes = align_up(raw);   // next job starts aligned
    if (raw > h->tcpack_bytes) return KFAC_ERR_WORKSPACE;
    if (used + raw > h->tcpack_bytes || (int)pr.size() == kMaxPackJobs)
      if (kfac_status e = flush()) return e;
    char* hi = h->ws + h->off_tcpack + used;
    char* lo = hi + (size_t)q.n * Kp * 4;
    used += bytes;
    PackJob j{};
    j.x = q.x;
    j.ld = q.ld;
    j.M = q.rows;
    j.d = q.d;
    j.n = q.n;
    j.Kp = Kp;
    j.hi = hi;
    j.lo = lo;
    pj.push_back(j);
    TcProblem t{};
    t.A = TcOperand{hi, lo, q.n, Kp};
    t.B = t.A;
    t.same_ab = true;
    t.upper = true;
    t.M = t.N = q.n;
    t.K = q.rows;
    t.e.alpha = q.alpha;
    t.e.beta = q.beta;
    t.e.C = q.F;
    t.e.ldc = q.n;
    t.layer = q.layer;
    t.kmode = q.kmode;
    pr.push_back(t);
  }
  return flush();
}

}  // namespace kfac
