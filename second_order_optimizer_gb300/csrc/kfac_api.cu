// Host side of the C ABI: argument checks, workspace layout, dispatch to the kernels.
#include "kfac_internal.cuh"
#include "syrk_simt.cuh"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <new>

namespace kfac {

static std::atomic<unsigned long long> g_launches{0};

int num_sms() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];   // 0: not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev < kMaxDev) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
    v = 1;
  if (dev < kMaxDev) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}
void count_launch(int n) { g_launches.fetch_add((unsigned long long)n); }
static std::atomic<int> g_last_cuda_error{0};

kfac_status check_launch() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return KFAC_OK;
  g_last_cuda_error.store((int)e);
  return KFAC_ERR_CUDA;
}

namespace {

bool valid_hp(const kfac_hparams* hp) {
  if (!hp) return false;
  if (!(hp->ema_decay >= 0.0 && hp->ema_decay < 1.0)) return false;
  if (!(hp->damping > 0.0) || !std::isfinite(hp->damping)) return false;
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->momentum) || !std::isfinite(hp->weight_decay))
    return false;
  if (hp->ema_init != KFAC_EMA_INIT_ZERO && hp->ema_init != KFAC_EMA_INIT_FIRST) return false;
  if (hp->math != KFAC_MATH_3XTF32 && hp->math != KFAC_MATH_BF16) return false;
  if (hp->ikfac != KFAC_IKFAC_OFF && hp->ikfac != KFAC_IKFAC_TF32 && hp->ikfac != KFAC_IKFAC_BF16)
    return false;
  return true;
}

bool valid_desc(const kfac_layer_desc& d) {
  if (d.kind != KFAC_KRON && d.kind != KFAC_DIAG) return false;
  if (d.d_out < 1 || d.d_in < 1 || (d.has_bias != 0 && d.has_bias != 1)) return false;
  if (d.in_dtype != KFAC_F32 && d.in_dtype != KFAC_BF16) return false;
  if (d.d_out > (1 << 20) || d.d_in > (1 << 20)) return false;
  return true;
}

struct Plan {
  std::vector<LayerInfo> layers;
  size_t off_status, off_part, part_floats, off_tickets, n_tickets, off_k4tmp, k4tmp_floats;
  size_t off_part_k4, off_tickets_k4;
  size_t off_k5part, k5part_floats, off_k5tickets, k5tickets_ints, off_invjobs, total;
  size_t off_tcpack, tcpack_bytes;
  size_t off_ones;
  int64_t ones_rows;
  int n_invjobs, max_kron_n;
};

bool make_plan(const kfac_layer_desc* descs, int nl, int64_t max_rows, const kfac_hparams* hp,
               Plan* P) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align_up(bytes ? bytes : 1);
    return o;
  };
  P->off_status = take(sizeof(DevStatus));
  P->layers.clear();
  size_t part = 0, tickets = 0, k4 = 0, k5 = 0, k5t = 0, tcpack = 0;
  size_t pack_sum = 0, k4_sum = 0, inv_pack_sum = 0;   // what a batch over every KRON layer would use
  int ninv = 0, maxn = 0;
  bool ones = false;   // a bf16 KRON layer whose bias column the direct SYRK reads as ones
  for (int i = 0; i < nl; ++i) {
    const kfac_layer_desc& d = descs[i];
    LayerInfo L{};
    L.kind = d.kind;
    L.o = d.d_out;
    L.d_in = d.d_in;
    L.n = d.d_in + d.has_bias;
    L.has_bias = d.has_bias;
    L.in_dtype = d.in_dtype;
    const size_t n = L.n, o = L.o, f = sizeof(float);
    L.m = take(o * n * f);
    if (d.kind == KFAC_KRON) {
      L.A = take(n * n * f);
      L.G = take(o * o * f);
      L.Ainv = take(n * n * f);
      L.Ginv = take(o * o * f);
      L.LA = take(n * n * f);
      L.LG = take(o * o * f);
      L.XA = take(n * n * f);
      L.XG = take(o * o * f);
      L.YA = take(inv_y_floats(L.n) * f);
      L.YG = take(inv_y_floats(L.o) * f);
      const size_t np = (size_t)tc_pitch(L.n, false), op = (size_t)tc_pitch(L.o, false);
      L.Ainv_hi = take(n * np * f);
      L.Ainv_lo = take(n * np * f);
      L.Ginv_hi = take(o * op * f);
      L.Ginv_lo = take(o * op * f);
      for (int w = 0; w < 2; ++w)
        for (int a = 0; a < 8; ++a)
          L.ik[w][a] = hp->ikfac ? take((w == 0 ? n * np : o * op) * f) : 0;
      size_t t1 = 0, t2 = 0;
      part = std::max(part, k1_scratch_floats(L.n, max_rows, &t1));
      part = std::max(part, k1_scratch_floats(L.o, max_rows, &t2));
      const bool bf = d.in_dtype == KFAC_BF16;
      ones = ones || (bf && d.has_bias && d.d_in % 64 == 0);
      part = std::max(part, tc_part_floats());
      // a batched group of one layer holds its A and G packs at once
      tcpack = std::max(tcpack, align_up(tc_pack_bytes(L.n, max_rows, bf)) +
                                    align_up(tc_pack_bytes(L.o, max_rows, bf)));
      // the inverse assembly packs X = L^{-1} (n x n, fp32) through the same buffer
      if (L.n >= kTcInverseMinN) {
        tcpack = std::max(tcpack, tc_pack_bytes(L.n, L.n, false));
        inv_pack_sum += align_up(tc_pack_bytes(L.n, L.n, false));
      }
      if (L.o >= kTcInverseMinN) {
        tcpack = std::max(tcpack, tc_pack_bytes(L.o, L.o, false));
        inv_pack_sum += align_up(tc_pack_bytes(L.o, L.o, false));
      }
      pack_sum += align_up(tc_pack_bytes(L.n, max_rows, bf)) + align_up(tc_pack_bytes(L.o, max_rows, bf));
      tickets = std::max({tickets, t1, t2, (size_t)16 * num_sms()});   // split-K: tile x cluster rank
      k4 = std::max(k4, 2 * o * np + 2 * n * op);
      // batched K4 aligns each of its four arrays (dW-hat and X^T halves) separately
      k4_sum += 2 * (align_up(o * np * sizeof(float)) + align_up(n * op * sizeof(float))) /
                sizeof(float);
      ninv += 4;   // three table sections: both factors, A only, G only
      maxn = std::max({maxn, L.n, L.o});
    } else {
      L.gs = take(o * f);
      L.as = take(n * f);
      L.ticket = take(sizeof(int));
    }
    k5 = std::max(k5, k5_scratch_floats(L.d_in + L.o, max_rows));
    k5t += (size_t)cdiv(L.d_in + L.o, 256);   // batched K5: every layer's column blocks
    P->layers.push_back(L);
  }
  // batched calls pack a group of layers at once, within a fixed budget
  tcpack = std::max(tcpack, std::min(pack_sum, kBatchScratchBudget));
  tcpack = std::max(tcpack, std::min(inv_pack_sum, kBatchScratchBudget));
  k4 = std::max(k4, std::min(k4_sum, kPrecondScratchBudget / sizeof(float)));
  P->part_floats = part;
  P->off_part = take(part * sizeof(float));
  P->n_tickets = tickets;
  P->off_tickets = take(tickets * sizeof(int));
  P->off_part_k4 = take(part * sizeof(float));
  P->off_tickets_k4 = take(tickets * sizeof(int));
  P->tcpack_bytes = tcpack;
  P->off_tcpack = take(tcpack);
  P->k4tmp_floats = k4;
  P->off_k4tmp = take(k4 * sizeof(float));
  P->ones_rows = ones ? max_rows : 0;
  P->off_ones = take((size_t)P->ones_rows * 64 * 2);
  // batched K5 spreads about 4 x SMs CTAs over the group, one part row per CTA
  k5 = std::max(k5, (size_t)256 * (4 * num_sms() + k5t));
  P->k5part_floats = k5;
  P->off_k5part = take(k5 * sizeof(float));
  P->off_k5tickets = take(k5t * sizeof(int));
  P->k5tickets_ints = k5t;
  P->off_invjobs = off;
  take(align_up(sizeof(InvJob) * ninv) + sizeof(SyrkJob) * ninv);
  P->n_invjobs = ninv;
  P->max_kron_n = maxn;
  P->total = off;
  return true;
}

kfac_status ensure_device(const kfac_ctx* h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KFAC_ERR_CUDA;
  if (dev != h->device && cudaSetDevice(h->device) != cudaSuccess) return KFAC_ERR_CUDA;
  return KFAC_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

kfac_status check_layer(const kfac_ctx* h, int layer, int kind) {
  if (!h) return KFAC_ERR_INVALID_ARG;
  if (layer < 0 || layer >= (int)h->layers.size()) return KFAC_ERR_INVALID_ARG;
  if (kind >= 0 && h->layers[layer].kind != kind) return KFAC_ERR_INVALID_ARG;
  return KFAC_OK;
}

kfac_status check_inputs(const kfac_ctx* h, const LayerInfo& L, const void* a, int64_t lda,
                         const void* g, int64_t ldg, int64_t rows) {
  const size_t es = L.in_dtype == KFAC_BF16 ? 2 : 4;
  if (!a || !g || !aligned(a, es) || !aligned(g, es)) return KFAC_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->max_rows) return KFAC_ERR_INVALID_ARG;
  if (lda < L.d_in || ldg < L.o) return KFAC_ERR_INVALID_ARG;
  return KFAC_OK;
}

}  // namespace

// The inversion job tables: section 0 holds A then G of every KRON layer,
// section 1 every A, section 2 every G, layers in order in each; a layer whose A
// is tied to another layer's contributes no A job.  Each InvJob has a parallel
// SyrkJob (the CUDA-core X^T X of the small factors).  Written to the host copy
// and, synchronously, to the device.
kfac_status write_inv_tables(kfac_ctx* h) {
  h->invjobs_host.clear();
  std::vector<SyrkJob> sj;
  auto add = [&](int i, int w) {
    const LayerInfo& L = h->layers[i];
    InvJob j{};
    const int n = w == 0 ? L.n : L.o;
    j.F = h->at<float>(w == 0 ? L.A : L.G);
    j.L = h->at<float>(w == 0 ? L.LA : L.LG);
    j.X = h->at<float>(w == 0 ? L.XA : L.XG);
    j.Y = h->at<float>(w == 0 ? L.YA : L.YG);
    j.Finv = h->at<float>(w == 0 ? L.Ainv : L.Ginv);
    j.Finv_hi = h->at<float>(w == 0 ? L.Ainv_hi : L.Ginv_hi);
    j.Finv_lo = h->at<float>(w == 0 ? L.Ainv_lo : L.Ginv_lo);
    if (h->hp.ikfac) {
      float** dst[8] = {&j.K_hi, &j.K_lo, &j.Kt_hi, &j.Kt_lo, &j.S1_hi, &j.S1_lo, &j.S2_hi, &j.S2_lo};
      for (int a = 0; a < 8; ++a) *dst[a] = h->at<float>(L.ik[w][a]);
    }
    j.n = n;
    j.np = (int)tc_pitch(n, false);
    j.layer = i;
    h->invjobs_host.push_back(j);
    SyrkJob s{};
    s.x = j.X;
    s.ld = n;
    s.M = n;
    s.d = n;
    s.n = n;
    s.has_bias = 0;
    s.x_lower = 1;
    s.alpha = 1.f;
    s.beta = 0.f;
    s.C = j.Finv;
    s.nt = (int)cdiv(n, SyrkTile::BM);
    s.splits = 1;
    s.rows_per_split = n;
    s.skip = n >= kTcInverseMinN ? 1 : 0;
    sj.push_back(s);
  };
  const int nl = (int)h->layers.size();
  const int masks[3] = {3, 1, 2};
  for (int sec = 0; sec < 3; ++sec) {
    h->tab_start[sec] = (int)h->invjobs_host.size();
    for (int i = 0; i < nl; ++i) {
      const LayerInfo& L = h->layers[i];
      if (L.kind != KFAC_KRON) continue;
      if ((masks[sec] & 1) && L.tied_to < 0) add(i, 0);
      if (masks[sec] & 2) add(i, 1);
    }
    h->tab_count[sec] = (int)h->invjobs_host.size() - h->tab_start[sec];
  }
  if ((int)h->invjobs_host.size() > h->n_invjobs) return KFAC_ERR_WORKSPACE;
  if (h->invjobs_host.empty()) return KFAC_OK;
  bool ok = cudaMemcpy(h->ws + h->off_invjobs, h->invjobs_host.data(),
                       sizeof(InvJob) * h->invjobs_host.size(), cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(h->ws + h->off_invjobs + align_up(sizeof(InvJob) * h->n_invjobs), sj.data(),
                        sizeof(SyrkJob) * sj.size(), cudaMemcpyHostToDevice) == cudaSuccess;
  return ok ? KFAC_OK : KFAC_ERR_CUDA;
}

namespace {

// Inputs of a KRON factor update: a and g each nullable (that factor is left
// as it is), not both; a tied layer takes no a.
kfac_status check_factor_inputs(const kfac_ctx* h, const LayerInfo& L, const void* a,
                                int64_t lda, const void* g, int64_t ldg, int64_t rows) {
  const size_t es = L.in_dtype == KFAC_BF16 ? 2 : 4;
  if (!a && !g) return KFAC_ERR_INVALID_ARG;
  if (a && (L.tied_to >= 0 || !aligned(a, es) || lda < L.d_in)) return KFAC_ERR_INVALID_ARG;
  if (g && (!aligned(g, es) || ldg < L.o)) return KFAC_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->max_rows) return KFAC_ERR_INVALID_ARG;
  return KFAC_OK;
}

// EMA weights of the old A and G for this update (0 for a factor's first update
// under EMA_INIT_FIRST), and the update counters afterwards.
void factor_decays(const kfac_ctx* h, const LayerInfo& L, float* da, float* dg) {
  const bool first_mode = h->hp.ema_init == KFAC_EMA_INIT_FIRST;
  *da = first_mode && L.t_a == 0 ? 0.f : (float)h->hp.ema_decay;
  *dg = first_mode && L.t_g == 0 ? 0.f : (float)h->hp.ema_decay;
}
// Both inverses a KRON layer preconditions with exist (a tied A: its source's).
bool has_inverses(const kfac_ctx* h, const LayerInfo& L) {
  const bool a = L.tied_to >= 0 ? h->layers[L.tied_to].inv_a : L.inv_a;
  return a && L.inv_g;
}
void count_updates(LayerInfo& L, const void* a, const void* g) {
  if (a) ++L.t_a;
  if (g) ++L.t_g;
}

// A convolution layer's NCHW inputs: geometry, sizes and alignment.
kfac_status check_conv(const kfac_ctx* h, const LayerInfo& L, const void* x, const void* gy,
                       const kfac_conv2d_geom& g, int64_t* rows) {
  const size_t es = L.in_dtype == KFAC_BF16 ? 2 : 4;
  if (!x && !gy) return KFAC_ERR_INVALID_ARG;
  if (x && (L.tied_to >= 0 || !aligned(x, es))) return KFAC_ERR_INVALID_ARG;
  if (gy && !aligned(gy, es)) return KFAC_ERR_INVALID_ARG;
  if (g.batch < 1 || g.in_channels < 1 || g.in_h < 1 || g.in_w < 1 || g.kernel_h < 1 ||
      g.kernel_w < 1 || g.stride_h < 1 || g.stride_w < 1 || g.pad_h < 0 || g.pad_w < 0 ||
      g.dilation_h < 1 || g.dilation_w < 1)
    return KFAC_ERR_INVALID_ARG;
  if ((int64_t)g.in_channels * g.kernel_h * g.kernel_w != L.d_in) return KFAC_ERR_INVALID_ARG;
  const int ho = conv_out(g.in_h, g.kernel_h, g.stride_h, g.pad_h, g.dilation_h);
  const int wo = conv_out(g.in_w, g.kernel_w, g.stride_w, g.pad_w, g.dilation_w);
  if (ho < 1 || wo < 1) return KFAC_ERR_INVALID_ARG;
  const int64_t lim = int64_t(1) << 31;
  const int64_t nx = (int64_t)g.batch * g.in_channels * g.in_h * g.in_w;
  const int64_t ny = (int64_t)g.batch * L.o * ho * wo;
  if (nx >= lim || ny >= lim) return KFAC_ERR_INVALID_ARG;
  const int64_t m = (int64_t)g.batch * ho * wo;
  if (m < 1 || m > h->max_rows) return KFAC_ERR_INVALID_ARG;
  *rows = m;
  return KFAC_OK;
}

}  // namespace
}  // namespace kfac

using namespace kfac;

extern "C" {

const char* kfac_status_string(kfac_status s) {
  switch (s) {
    case KFAC_OK: return "ok";
    case KFAC_ERR_INVALID_ARG: return "invalid argument";
    case KFAC_ERR_WORKSPACE: return "workspace too small or misaligned";
    case KFAC_ERR_STATE: return "call out of order (e.g. precondition before invert)";
    case KFAC_ERR_NOT_PD: return "damped factor is not positive definite";
    case KFAC_ERR_TIMEOUT: return "device pipeline wait timed out";
    case KFAC_ERR_CUDA: return "CUDA runtime error";
    case KFAC_ERR_UNSUPPORTED: return "unsupported by the library";
  }
  return "unknown status";
}

unsigned long long kfac_launch_count(void) { return g_launches.load(); }

const char* kfac_last_cuda_error(void) {
  return cudaGetErrorString((cudaError_t)g_last_cuda_error.load());
}

kfac_status kfac_workspace_size(const kfac_layer_desc* layers, int n_layers,
                                const kfac_hparams* hp, int64_t max_rows, size_t* bytes) {
  if (!layers || n_layers < 1 || !bytes || max_rows < 1 || !valid_hp(hp))
    return KFAC_ERR_INVALID_ARG;
  for (int i = 0; i < n_layers; ++i)
    if (!valid_desc(layers[i])) return KFAC_ERR_INVALID_ARG;
  Plan P;
  make_plan(layers, n_layers, max_rows, hp, &P);
  *bytes = P.total;
  return KFAC_OK;
}

kfac_status kfac_create(const kfac_layer_desc* layers, int n_layers, const kfac_hparams* hp,
                        int64_t max_rows, void* d_workspace, size_t bytes, kfac_handle* out) {
  if (!out) return KFAC_ERR_INVALID_ARG;
  *out = nullptr;
  size_t need = 0;
  if (kfac_status e = kfac_workspace_size(layers, n_layers, hp, max_rows, &need)) return e;
  if (!d_workspace || !aligned(d_workspace, kAlign) || bytes < need) return KFAC_ERR_WORKSPACE;
  Plan P;
  make_plan(layers, n_layers, max_rows, hp, &P);
  kfac_ctx* h = new (std::nothrow) kfac_ctx();
  if (!h) return KFAC_ERR_INVALID_ARG;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return KFAC_ERR_CUDA;
  }
  h->hp = *hp;
  h->max_rows = max_rows;
  h->ws = static_cast<char*>(d_workspace);
  h->ws_bytes = bytes;
  h->layers = P.layers;
  h->off_status = P.off_status;
  h->off_part = P.off_part;
  h->part_floats = P.part_floats;
  h->off_tickets = P.off_tickets;
  h->n_tickets = P.n_tickets;
  h->off_part_k4 = P.off_part_k4;
  h->off_tickets_k4 = P.off_tickets_k4;
  h->off_tcpack = P.off_tcpack;
  h->tcpack_bytes = P.tcpack_bytes;
  h->off_ones = P.off_ones;
  h->ones_rows = P.ones_rows;
  h->off_k4tmp = P.off_k4tmp;
  h->k4tmp_floats = P.k4tmp_floats;
  h->off_k5part = P.off_k5part;
  h->k5part_floats = P.k5part_floats;
  h->off_k5tickets = P.off_k5tickets;
  h->k5tickets_ints = P.k5tickets_ints;
  h->off_invjobs = P.off_invjobs;
  h->n_invjobs = P.n_invjobs;
  h->max_kron_n = P.max_kron_n;
  if (P.n_invjobs > 0) {
    if (cudaStreamCreateWithFlags(&h->side_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_panel, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_rest, cudaEventDisableTiming) != cudaSuccess) {
      kfac_destroy(h);
      return KFAC_ERR_CUDA;
    }
  }
  bool ok = cudaMemset(d_workspace, 0, need) == cudaSuccess;
  if (h->ones_rows > 0) {   // bf16 1.0 = 0x3f80 in the first element of each 128-byte row
    char* o = h->ws + h->off_ones;
    ok = ok && cudaMemset2D(o, 128, 0x80, 1, (size_t)h->ones_rows) == cudaSuccess;
    ok = ok && cudaMemset2D(o + 1, 128, 0x3f, 1, (size_t)h->ones_rows) == cudaSuccess;
  }
  ok = ok && write_inv_tables(h) == KFAC_OK;
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    kfac_destroy(h);
    return KFAC_ERR_CUDA;
  }
  *out = h;
  return KFAC_OK;
}

kfac_status kfac_set_hparams(kfac_handle h, const kfac_hparams* hp) {
  if (!h || !valid_hp(hp)) return KFAC_ERR_INVALID_ARG;
  if (hp->ikfac != h->hp.ikfac) return KFAC_ERR_INVALID_ARG;   // fixed at creation
  if (hp->math != h->hp.math) return KFAC_ERR_INVALID_ARG;     // the inverses' storage form
  h->hp = *hp;
  return KFAC_OK;
}

kfac_status kfac_update_factors(kfac_handle h, int layer, const void* a, int64_t lda,
                                const void* g, int64_t ldg, int64_t rows, double scale,
                                cudaStream_t stream) {
  if (kfac_status e = check_layer(h, layer, KFAC_KRON)) return e;
  LayerInfo& L = h->layers[layer];
  if (kfac_status e = check_factor_inputs(h, L, a, lda, g, ldg, rows)) return e;
  if (!std::isfinite(scale)) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  float da, dg;
  factor_decays(h, L, &da, &dg);
  kfac_status e = launch_update_factors(h, layer, a, lda, g, ldg, rows, scale, da, dg, stream);
  if (e == KFAC_OK) count_updates(L, a, g);
  return e;
}

kfac_status kfac_update_factors_batched(kfac_handle h, int count, const int* layers,
                                        const void* const* a, const int64_t* lda,
                                        const void* const* g, const int64_t* ldg,
                                        const int64_t* rows, double scale, cudaStream_t stream) {
  if (!h || count < 1 || !layers || !a || !lda || !g || !ldg || !rows || !std::isfinite(scale))
    return KFAC_ERR_INVALID_ARG;
  std::vector<char> seen(h->layers.size(), 0);
  for (int i = 0; i < count; ++i) {
    if (kfac_status e = check_layer(h, layers[i], KFAC_KRON)) return e;
    if (seen[layers[i]]++) return KFAC_ERR_INVALID_ARG;   // a layer at most once per batch
    const LayerInfo& L = h->layers[layers[i]];
    if (L.in_dtype != h->layers[layers[0]].in_dtype) return KFAC_ERR_INVALID_ARG;
    if (kfac_status e = check_factor_inputs(h, L, a[i], lda[i], g[i], ldg[i], rows[i])) return e;
  }
  if (kfac_status e = ensure_device(h)) return e;
  std::vector<float> da(count), dg(count);
  for (int i = 0; i < count; ++i) factor_decays(h, h->layers[layers[i]], &da[i], &dg[i]);
  kfac_status e = launch_update_factors_batched(h, count, layers, a, lda, g, ldg, rows, scale,
                                                da.data(), dg.data(), stream);
  if (e == KFAC_OK)
    for (int i = 0; i < count; ++i) count_updates(h->layers[layers[i]], a[i], g[i]);
  return e;
}

kfac_status kfac_update_factors_conv2d_batched(kfac_handle h, int count, const int* layers,
                                               const void* const* x, const void* const* gy,
                                               const kfac_conv2d_geom* geoms, double scale,
                                               cudaStream_t stream) {
  if (!h || count < 1 || !layers || !x || !gy || !geoms || !std::isfinite(scale))
    return KFAC_ERR_INVALID_ARG;
  std::vector<char> seen(h->layers.size(), 0);
  std::vector<int64_t> rows(count);
  for (int i = 0; i < count; ++i) {
    if (kfac_status e = check_layer(h, layers[i], KFAC_KRON)) return e;
    if (seen[layers[i]]++) return KFAC_ERR_INVALID_ARG;
    const LayerInfo& L = h->layers[layers[i]];
    if (L.in_dtype != h->layers[layers[0]].in_dtype) return KFAC_ERR_INVALID_ARG;
    if (kfac_status e = check_conv(h, L, x[i], gy[i], geoms[i], &rows[i])) return e;
  }
  if (kfac_status e = ensure_device(h)) return e;
  std::vector<float> da(count), dg(count);
  for (int i = 0; i < count; ++i) factor_decays(h, h->layers[layers[i]], &da[i], &dg[i]);
  kfac_status e = launch_update_factors_batched(h, count, layers, x, nullptr, gy, nullptr,
                                                rows.data(), scale, da.data(), dg.data(), stream,
                                                geoms);
  if (e == KFAC_OK)
    for (int i = 0; i < count; ++i) count_updates(h->layers[layers[i]], x[i], gy[i]);
  return e;
}

kfac_status kfac_update_factors_conv2d(kfac_handle h, int layer, const void* x, const void* gy,
                                       const kfac_conv2d_geom* geom, double scale,
                                       cudaStream_t stream) {
  if (!geom) return KFAC_ERR_INVALID_ARG;
  return kfac_update_factors_conv2d_batched(h, 1, &layer, &x, &gy, geom, scale, stream);
}

kfac_status kfac_diag_factors(kfac_handle h, int layer, const void* a, int64_t lda,
                              const void* g, int64_t ldg, int64_t rows, double scale,
                              float* g_new, float* a_new, cudaStream_t stream) {
  if (kfac_status e = check_layer(h, layer, -1)) return e;
  const LayerInfo& L = h->layers[layer];
  if (kfac_status e = check_inputs(h, L, a, lda, g, ldg, rows)) return e;
  if (!g_new || !a_new || !aligned(g_new, 4) || !aligned(a_new, 4)) return KFAC_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  return launch_diag_factors(h, layer, a, lda, g, ldg, rows, scale, g_new, a_new, stream);
}

kfac_status kfac_diag_factors_conv2d(kfac_handle h, int layer, const void* x, const void* gy,
                                     const kfac_conv2d_geom* geom, double scale,
                                     float* g_new, float* a_new, cudaStream_t stream) {
  if (kfac_status e = check_layer(h, layer, -1)) return e;
  const LayerInfo& L = h->layers[layer];
  if (!geom || !x || !gy || !std::isfinite(scale)) return KFAC_ERR_INVALID_ARG;
  if (!g_new || !a_new || !aligned(g_new, 4) || !aligned(a_new, 4)) return KFAC_ERR_INVALID_ARG;
  int64_t rows = 0;
  if (kfac_status e = check_conv(h, L, x, gy, *geom, &rows)) return e;
  if (kfac_status e = ensure_device(h)) return e;
  return launch_diag_factors_conv(h, layer, x, gy, *geom, scale, g_new, a_new, stream);
}

kfac_status kfac_diag_factors_batched(kfac_handle h, int count, const int* layers,
                                      const void* const* a, const int64_t* lda,
                                      const void* const* g, const int64_t* ldg,
                                      const int64_t* rows, double scale, float* const* g_new,
                                      float* const* a_new, cudaStream_t stream) {
  if (!h || count < 1 || !layers || !a || !lda || !g || !ldg || !rows || !g_new || !a_new ||
      !std::isfinite(scale))
    return KFAC_ERR_INVALID_ARG;
  std::vector<char> seen(h->layers.size(), 0);
  for (int i = 0; i < count; ++i) {
    if (kfac_status e = check_layer(h, layers[i], -1)) return e;
    if (seen[layers[i]]++) return KFAC_ERR_INVALID_ARG;
    const LayerInfo& L = h->layers[layers[i]];
    if (L.in_dtype != h->layers[layers[0]].in_dtype) return KFAC_ERR_INVALID_ARG;
    if (kfac_status e = check_inputs(h, L, a[i], lda[i], g[i], ldg[i], rows[i])) return e;
    if (!g_new[i] || !a_new[i] || !aligned(g_new[i], 4) || !aligned(a_new[i], 4))
      return KFAC_ERR_INVALID_ARG;
  }
  if (kfac_status e = ensure_device(h)) return e;
  return launch_diag_factors_batched(h, count, layers, a, lda, g, ldg, rows, scale, g_new, a_new,
                                     stream);
}

kfac_status kfac_invert_factors(kfac_handle h, int layer, int which, cudaStream_t stream) {
  if (!h || which < 1 || which > 3) return KFAC_ERR_INVALID_ARG;
  if (layer != -1 && check_layer(h, layer, KFAC_KRON) != KFAC_OK) return KFAC_ERR_INVALID_ARG;
  if (h->n_invjobs == 0) return layer == -1 ? KFAC_OK : KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  kfac_status e = launch_invert(h, layer, which, stream);
  if (e != KFAC_OK) return e;
  for (int i = 0; i < (int)h->layers.size(); ++i) {
    LayerInfo& L = h->layers[i];
    if (L.kind != KFAC_KRON || (layer != -1 && layer != i)) continue;
    if ((which & KFAC_FACTOR_A) && L.tied_to < 0) L.inv_a = true;
    if (which & KFAC_FACTOR_G) L.inv_g = true;
  }
  return KFAC_OK;
}

kfac_status kfac_ikfac_update(kfac_handle h, int layer, double beta, cudaStream_t stream) {
  if (!h) return KFAC_ERR_INVALID_ARG;
  if (!h->hp.ikfac) return KFAC_ERR_UNSUPPORTED;
  if (!(beta > 0.0 && beta < 2.0)) return KFAC_ERR_INVALID_ARG;
  if (layer != -1 && check_layer(h, layer, KFAC_KRON) != KFAC_OK) return KFAC_ERR_INVALID_ARG;
  if (h->n_invjobs == 0) return layer == -1 ? KFAC_OK : KFAC_ERR_INVALID_ARG;
  for (int i = 0; i < (int)h->layers.size(); ++i) {
    const LayerInfo& L = h->layers[i];
    if (L.kind != KFAC_KRON || (layer != -1 && layer != i)) continue;
    if (!has_inverses(h, L)) return KFAC_ERR_STATE;   // K is seeded by kfac_invert
  }
  if (kfac_status e = ensure_device(h)) return e;
  return launch_ikfac_update(h, layer, (float)beta, stream);
}

kfac_status kfac_invert(kfac_handle h, int layer, cudaStream_t stream) {
  return kfac_invert_factors(h, layer, KFAC_FACTOR_A | KFAC_FACTOR_G, stream);
}

kfac_status kfac_tie_a_factor(kfac_handle h, int layer, int source) {
  if (!h || layer == source) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = check_layer(h, layer, KFAC_KRON)) return e;
  if (kfac_status e = check_layer(h, source, KFAC_KRON)) return e;
  LayerInfo& L = h->layers[layer];
  const LayerInfo& S = h->layers[source];
  if (L.n != S.n || S.tied_to >= 0 || L.tied_to >= 0) return KFAC_ERR_INVALID_ARG;
  for (const LayerInfo& X : h->layers)
    if (X.tied_to == layer) return KFAC_ERR_INVALID_ARG;    // no chains
  if (L.t_a || L.t_g || L.inv_a || L.inv_g || S.t_a || S.t_g || S.inv_a || S.inv_g)
    return KFAC_ERR_STATE;
  if (kfac_status e = ensure_device(h)) return e;
  L.tied_to = source;
  L.A = S.A;
  L.LA = S.LA;
  L.XA = S.XA;
  L.YA = S.YA;
  L.Ainv = S.Ainv;
  L.Ainv_hi = S.Ainv_hi;
  L.Ainv_lo = S.Ainv_lo;
  for (int a = 0; a < 8; ++a) L.ik[0][a] = S.ik[0][a];
  kfac_status e = write_inv_tables(h);
  if (e == KFAC_OK && cudaDeviceSynchronize() != cudaSuccess) e = KFAC_ERR_CUDA;
  return e;
}

kfac_status kfac_precondition(kfac_handle h, int layer, const float* grad_w, int64_t ldgw,
                              const float* grad_b, float* out_w, float* out_b, float* param_w,
                              float* param_b, cudaStream_t stream) {
  if (kfac_status e = check_layer(h, layer, KFAC_KRON)) return e;
  const LayerInfo& L = h->layers[layer];
  if (!grad_w || !aligned(grad_w, 4) || ldgw < L.d_in) return KFAC_ERR_INVALID_ARG;
  if (L.has_bias && !grad_b) return KFAC_ERR_INVALID_ARG;
  if (!out_w && !param_w) return KFAC_ERR_INVALID_ARG;
  if (L.has_bias && out_w && !out_b) return KFAC_ERR_INVALID_ARG;
  if (L.has_bias && param_w && !param_b) return KFAC_ERR_INVALID_ARG;
  if (!has_inverses(h, L)) return KFAC_ERR_STATE;
  if (kfac_status e = ensure_device(h)) return e;
  return launch_precondition(h, layer, grad_w, ldgw, L.has_bias ? grad_b : nullptr, out_w,
                             L.has_bias ? out_b : nullptr, param_w,
                             L.has_bias ? param_b : nullptr, stream);
}

kfac_status kfac_precondition_batched(kfac_handle h, int count, const int* layers,
                                      const float* const* grad_w, const int64_t* ldgw,
                                      const float* const* grad_b, float* const* out_w,
                                      float* const* out_b, float* const* param_w,
                                      float* const* param_b, cudaStream_t stream) {
  if (!h || count < 1 || !layers || !grad_w || !ldgw || (!out_w && !param_w))
    return KFAC_ERR_INVALID_ARG;
  std::vector<char> seen(h->layers.size(), 0);
  std::vector<const float*> gb(count, nullptr);
  std::vector<float*> ob(count, nullptr), pb(count, nullptr);
  for (int i = 0; i < count; ++i) {
    if (kfac_status e = check_layer(h, layers[i], KFAC_KRON)) return e;
    if (seen[layers[i]]++) return KFAC_ERR_INVALID_ARG;
    const LayerInfo& L = h->layers[layers[i]];
    const float* bw = grad_b ? grad_b[i] : nullptr;
    float* o_w = out_w ? out_w[i] : nullptr;
    float* o_b = out_b ? out_b[i] : nullptr;
    float* p_w = param_w ? param_w[i] : nullptr;
    float* p_b = param_b ? param_b[i] : nullptr;
    if (!grad_w[i] || !aligned(grad_w[i], 4) || ldgw[i] < L.d_in) return KFAC_ERR_INVALID_ARG;
    if (L.has_bias && !bw) return KFAC_ERR_INVALID_ARG;
    if (!o_w && !p_w) return KFAC_ERR_INVALID_ARG;
    if (L.has_bias && o_w && !o_b) return KFAC_ERR_INVALID_ARG;
    if (L.has_bias && p_w && !p_b) return KFAC_ERR_INVALID_ARG;
    if (!has_inverses(h, L)) return KFAC_ERR_STATE;
    gb[i] = L.has_bias ? bw : nullptr;
    ob[i] = L.has_bias ? o_b : nullptr;
    pb[i] = L.has_bias ? p_b : nullptr;
  }
  if (kfac_status e = ensure_device(h)) return e;
  return launch_precondition_batched(h, count, layers, grad_w, ldgw, gb.data(), out_w, ob.data(),
                                     param_w, pb.data(), stream);
}

kfac_status kfac_diag_step(kfac_handle h, int layer, const float* g_new, const float* a_new,
                           const float* grad_w, const float* grad_b, float* param_w,
                           float* param_b, float* out_w, float* out_b, cudaStream_t stream) {
  if (kfac_status e = check_layer(h, layer, KFAC_DIAG)) return e;
  LayerInfo& L = h->layers[layer];
  if (!g_new || !a_new || !grad_w || !param_w) return KFAC_ERR_INVALID_ARG;
  if (L.has_bias && (!grad_b || !param_b)) return KFAC_ERR_INVALID_ARG;
  if (L.has_bias && out_w && !out_b) return KFAC_ERR_INVALID_ARG;
  for (const void* p : {(const void*)g_new, (const void*)a_new, (const void*)grad_w,
                        (const void*)param_w})
    if (!aligned(p, 4)) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  const bool first = L.t_diag == 0 && h->hp.ema_init == KFAC_EMA_INIT_FIRST;
  const float decay = first ? 0.f : (float)h->hp.ema_decay;
  kfac_status e = launch_diag_step(h, layer, decay, g_new, a_new, grad_w,
                                   L.has_bias ? grad_b : nullptr, param_w,
                                   L.has_bias ? param_b : nullptr, out_w,
                                   L.has_bias ? out_b : nullptr, stream);
  if (e == KFAC_OK) ++L.t_diag;
  return e;
}

kfac_status kfac_diag_step_batched(kfac_handle h, int count, const int* layers,
                                   const float* const* g_new, const float* const* a_new,
                                   const float* const* grad_w, const float* const* grad_b,
                                   float* const* param_w, float* const* param_b,
                                   float* const* out_w, float* const* out_b,
                                   cudaStream_t stream) {
  if (!h || count < 1 || !layers || !g_new || !a_new || !grad_w || !param_w)
    return KFAC_ERR_INVALID_ARG;
  std::vector<char> seen(h->layers.size(), 0);
  std::vector<const float*> gb(count, nullptr);
  std::vector<float*> pb(count, nullptr), ow(count, nullptr), ob(count, nullptr);
  std::vector<float> decay(count);
  for (int i = 0; i < count; ++i) {
    if (kfac_status e = check_layer(h, layers[i], KFAC_DIAG)) return e;
    if (seen[layers[i]]++) return KFAC_ERR_INVALID_ARG;
    const LayerInfo& L = h->layers[layers[i]];
    const float* b_g = grad_b ? grad_b[i] : nullptr;
    float* b_p = param_b ? param_b[i] : nullptr;
    float* w_o = out_w ? out_w[i] : nullptr;
    float* b_o = out_b ? out_b[i] : nullptr;
    if (!g_new[i] || !a_new[i] || !grad_w[i] || !param_w[i]) return KFAC_ERR_INVALID_ARG;
    if (L.has_bias && (!b_g || !b_p)) return KFAC_ERR_INVALID_ARG;
    if (L.has_bias && w_o && !b_o) return KFAC_ERR_INVALID_ARG;
    for (const void* p : {(const void*)g_new[i], (const void*)a_new[i], (const void*)grad_w[i],
                          (const void*)param_w[i]})
      if (!aligned(p, 4)) return KFAC_ERR_INVALID_ARG;
    gb[i] = L.has_bias ? b_g : nullptr;
    pb[i] = L.has_bias ? b_p : nullptr;
    ow[i] = w_o;
    ob[i] = L.has_bias ? b_o : nullptr;
    const bool first = L.t_diag == 0 && h->hp.ema_init == KFAC_EMA_INIT_FIRST;
    decay[i] = first ? 0.f : (float)h->hp.ema_decay;
  }
  if (kfac_status e = ensure_device(h)) return e;
  kfac_status e = launch_diag_step_batched(h, count, layers, decay.data(), g_new, a_new, grad_w,
                                           gb.data(), param_w, pb.data(), ow.data(), ob.data(),
                                           stream);
  if (e == KFAC_OK)
    for (int i = 0; i < count; ++i) ++h->layers[layers[i]].t_diag;
  return e;
}

kfac_status kfac_selftest_timeout(kfac_handle h, int64_t wait_cycles, cudaStream_t stream) {
  if (!h || wait_cycles < 1 || wait_cycles > (int64_t(1) << 31)) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  return launch_wait_selftest(h, wait_cycles, stream);
}

kfac_status kfac_get_status(kfac_handle h, int* bad_layer, int* info) {
  if (!h) return KFAC_ERR_INVALID_ARG;
  if (kfac_status e = ensure_device(h)) return e;
  if (cudaDeviceSynchronize() != cudaSuccess) return KFAC_ERR_CUDA;
  DevStatus s{};
  if (cudaMemcpy(&s, h->status(), sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KFAC_ERR_CUDA;
  if (bad_layer) *bad_layer = s.code ? s.layer : -1;
  if (info) *info = s.code ? s.info : 0;
  if (s.code) {
    if (cudaMemset(h->status(), 0, sizeof(DevStatus)) != cudaSuccess) return KFAC_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return KFAC_ERR_CUDA;
  }
  return (kfac_status)s.code;
}

kfac_status kfac_state_info(kfac_handle h, int layer, int which, size_t* offset, size_t* bytes) {
  if (check_layer(h, layer, -1) != KFAC_OK || !offset || !bytes) return KFAC_ERR_INVALID_ARG;
  const LayerInfo& L = h->layers[layer];
  const size_t f = sizeof(float), n = L.n, o = L.o;
  const bool kron = L.kind == KFAC_KRON;
  switch (which) {
    case KFAC_STATE_A: if (!kron) return KFAC_ERR_INVALID_ARG; *offset = L.A; *bytes = n * n * f; break;
    case KFAC_STATE_G: if (!kron) return KFAC_ERR_INVALID_ARG; *offset = L.G; *bytes = o * o * f; break;
    case KFAC_STATE_AINV: if (!kron) return KFAC_ERR_INVALID_ARG; *offset = L.Ainv; *bytes = n * n * f; break;
    case KFAC_STATE_GINV: if (!kron) return KFAC_ERR_INVALID_ARG; *offset = L.Ginv; *bytes = o * o * f; break;
    case KFAC_STATE_MOMENTUM: *offset = L.m; *bytes = o * n * f; break;
    case KFAC_STATE_GDIAG: if (kron) return KFAC_ERR_INVALID_ARG; *offset = L.gs; *bytes = o * f; break;
    case KFAC_STATE_ADIAG: if (kron) return KFAC_ERR_INVALID_ARG; *offset = L.as; *bytes = n * f; break;
    default: return KFAC_ERR_INVALID_ARG;
  }
  return KFAC_OK;
}

kfac_status kfac_destroy(kfac_handle h) {
  if (!h) return KFAC_ERR_INVALID_ARG;
  if (h->side_stream) cudaStreamDestroy(h->side_stream);
  if (h->ev_panel) cudaEventDestroy(h->ev_panel);
  if (h->ev_rest) cudaEventDestroy(h->ev_rest);
  delete h;
  return KFAC_OK;
}

}  // extern "C"
