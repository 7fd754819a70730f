// Host layer of the fused linear cross-entropy library: argument checks,
// workspace carving, TMA tensor maps, work decomposition and the launch
// sequence behind the C ABI declared in include/lce.h.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/lce.h"
#include "lce_internal.h"

namespace lce {

// The device error word: kernels OR error bits into it, lce_get_error reads
// and clears it. One per device (module globals are per device).
__device__ unsigned g_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 16;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

thread_local char t_last_cuda_error[256] = "";

lce_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(t_last_cuda_error, sizeof t_last_cuda_error, "%s: %s", where,
                cudaGetErrorString(e));
  return LCE_ERR_CUDA;
}

// ---- optional per-kernel timing (lce_profile_start / lce_profile_stop) ----
// When on, every kernel this thread launches is bracketed by two CUDA events
// on its stream; stop() waits for them and sums durations per kernel kind.
const char* const kKindNames[LCE_KERNEL_KINDS] = {
    "count_valid",  "gemm_lse",     "lse_combine",   "loss_finalize",
    "f32_to_bf16",  "gemm_grad",    "gemm_dH",       "gemm_dW",
    "test_gemm",    "wait_probe",   "gemm_fused",    "grad_from_exp",
    "scale_grads",  "mlp_gate_up",  "mlp_down",      "mlp_da",
    "mlp_dx",       "mlp_dWd",      "mlp_dWgu",      "slice_stats",
    "combine_slices", "shard_combine"};

struct ProfRec {
  int kind;
  cudaEvent_t e0, e1;
  double flops;
};

struct Profiler {
  bool on = false;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  cudaEvent_t take() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
};
thread_local Profiler t_prof;

// Brackets one launch: construct before, call done(flops) after.
struct ProfScope {
  int kind;
  cudaStream_t s;
  cudaEvent_t e0 = nullptr;
  ProfScope(int k, cudaStream_t st) : kind(k), s(st) {
    if (t_prof.on && (e0 = t_prof.take()) != nullptr) cudaEventRecord(e0, s);
  }
  void done(double flops) {
    if (!e0) return;
    cudaEvent_t e1 = t_prof.take();
    if (!e1) return;
    cudaEventRecord(e1, s);
    t_prof.recs.push_back({kind, e0, e1, flops});
  }
};

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int pair_slots = 0;       // co-resident CTA pairs of the pair kernels
  unsigned* err = nullptr;  // device address of g_error_word
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

// The driver calls a launch makes (tensor-map encoding) need a CUDA context
// current on the calling thread. A thread that has made no runtime call yet
// (for instance an autograd worker whose framework skipped setting the
// device it already reported) may have none; the runtime would make its
// device's primary context current at its first call that needs one, so do
// that here, and only then (a context the caller made current is kept).
lce_status ensure_context() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext ctx = nullptr;
  if (get_current && get_current(&ctx) == CUDA_SUCCESS && ctx) return LCE_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "cudaSetDevice");
}

lce_status device_info(DeviceInfo** out) {
  const lce_status cs = ensure_context();
  if (cs != LCE_OK) return cs;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.num_sms,
                                    cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    // The kernels are built for sm_103a only.
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress");
      d.err = static_cast<unsigned*>(p);
      if ((e = pair_max_active_clusters(&d.pair_slots)) != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
    }
    d.ready = true;
  }
  if (!d.supported) return LCE_ERR_UNSUPPORTED;
  *out = &d;
  return LCE_OK;
}

// Contractions on single CTAs (128 x 256 tiles) or on CTA pairs
// (256 x 256 tiles, tcgen05 cta_group::2). LCE_CTA_PAIR=0/1 in the
// environment or lce_set_cta_pair() choose; the default is kDefaultPair.
constexpr int kDefaultPair = 1;
std::atomic<int> g_pair_mode{-1};

bool use_pair() {
  int v = g_pair_mode.load();
  if (v < 0) {
    const char* s = std::getenv("LCE_CTA_PAIR");
    v = (s && *s) ? (std::atoi(s) != 0) : kDefaultPair;
    g_pair_mode.store(v);
  }
  return v != 0;
}

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("LCE_WAIT_TIMEOUT_MS");
    if (s && *s) {
      const double ms = std::atof(s);
      if (ms > 0) return static_cast<uint64_t>(ms * 1e6);
    }
    return kDefaultTimeoutNs;
  }();
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// rows `row_bytes` apart; boxes of box_inner x box_outer with 128-byte
// swizzle (box_inner = 64 elements = one swizzle row). Out-of-range
// elements of a box read as zero.
lce_status make_tmap(CUtensorMap* tm, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                     uint32_t box_outer,
                     CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tmap_encoder();
  if (!enc) {
    std::snprintf(t_last_cuda_error, sizeof t_last_cuda_error,
                  "cuTensorMapEncodeTiled not available");
    return LCE_ERR_CUDA;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_cuda_error, sizeof t_last_cuda_error,
                  "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, "
                  "stride %llu",
                  static_cast<int>(r), static_cast<unsigned long long>(inner),
                  static_cast<unsigned long long>(outer),
                  static_cast<unsigned long long>(row_bytes));
    return LCE_ERR_CUDA;
  }
  return LCE_OK;
}

// Tensor maps of the two operand layouts the contractions read.
// K-major: rows of the operand's M (or N) index, K contiguous; one box per
// stage covers the whole 64-wide K slice of `rows_per_box` rows.
lce_status tmap_kmajor(CUtensorMap* tm, const void* base, int64_t k_extent,
                       int64_t rows, int64_t row_elems, uint32_t rows_per_box) {
  return make_tmap(tm, base, k_extent, rows, row_elems * 2, BK, rows_per_box);
}
// MN-major: rows of K, the operand's M (or N) index contiguous; boxes of
// 64 MN x 64 K, several per stage.
lce_status tmap_mnmajor(CUtensorMap* tm, const void* base, int64_t mn_extent,
                        int64_t k_rows, int64_t row_elems) {
  return make_tmap(tm, base, mn_extent, k_rows, row_elems * 2, 64, BK);
}

// Store map of a bf16 [rows][row_elems] matrix of `cols` valid columns, in
// the 32-row x 32-column boxes (64 bytes per row, 64-byte swizzle) that an
// epilogue warp stages in shared memory (EPI_BOX).
lce_status tmap_store_box(CUtensorMap* tm, const void* base, int64_t cols,
                          int64_t rows, int64_t row_elems) {
  return make_tmap(tm, base, cols, rows, row_elems * 2, EPI_BOX, EPI_BOX,
                   CU_TENSOR_MAP_SWIZZLE_64B);
}

// ---- the contractions' tile order --------------------------------------------
// The vocabulary sweeps (forward logits and their recompute) take enough
// column-tile runs per row block that at most this many bytes of A row
// panels are live at once; they stay in L2 while every CTA sweeps W.
constexpr double kL2PanelBudget = 48e6;

// Every other contraction (one output tile per work unit) walks its tiles
// in groups of kGroupN column tiles, the row blocks varying inside a group,
// so a wave of 76 pair tiles spans about 9.5 row blocks x 8 column panels
// instead of the row-major order's 76 / num_n row blocks x num_n columns,
// and reads fewer distinct operand panels from DRAM. On the 8B shard this
// cut each launch's DRAM reads from 30.3 to 25.5 GB (dH) and from 32.2 to
// 27.3 GB (dW); on the gated MLP's contractions, with pacing, from ~95 to
// ~31 GB per row chunk. The tile order changes no result: every tile is
// computed by the same arithmetic wherever it sits in the order.
constexpr int kGroupN = 8;

// Wave pacing of the contractions (GemmGeom::wave_ctr): on unless
// LCE_WAVE_SYNC=0 or lce_set_wave_sync(0).
std::atomic<int> g_wave_mode{-1};

bool wave_sync_on() {
  int v = g_wave_mode.load();
  if (v < 0) {
    const char* env = std::getenv("LCE_WAVE_SYNC");
    v = (env && *env) ? (std::atoi(env) != 0) : 1;
    g_wave_mode.store(v);
  }
  return v != 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Column-tile runs per row block for the contractions that sweep the whole
// vocabulary (forward logits and their backward recompute). Enough runs that
// at most ~48 MB of A row panels are live at once (they stay in L2 while
// every CTA sweeps W), then the smallest count whose static schedule is
// within 5% of the best one.
void choose_splits(int num_m, int num_n, int nsm, int64_t K, int* splits,
                   int* tps, int rows_per_unit = BM) {
  const double panel = static_cast<double>(rows_per_unit) * K * 2.0;
  int s_min = static_cast<int>(std::ceil(nsm * panel / kL2PanelBudget));
  const int s_max = std::max(1, std::min(kMaxSplits, num_n));
  s_min = std::max(1, std::min(s_min, s_max));
  const double work = static_cast<double>(num_m) * num_n;
  double best = -1.0;
  double effs[kMaxSplits + 1] = {0};
  for (int s = s_min; s <= s_max; ++s) {
    const int t = static_cast<int>(ceil_div(num_n, s));
    const int se = static_cast<int>(ceil_div(num_n, t));
    const double units = static_cast<double>(num_m) * se;
    const double makespan = std::ceil(units / nsm) * t;
    effs[s] = work / (makespan * nsm);
    best = std::max(best, effs[s]);
  }
  for (int s = s_min; s <= s_max; ++s) {
    if (effs[s] >= 0.95 * best) {
      *tps = static_cast<int>(ceil_div(num_n, s));
      *splits = static_cast<int>(ceil_div(num_n, *tps));
      return;
    }
  }
  *tps = num_n;
  *splits = 1;
}

GemmGeom make_geom(int64_t M, int64_t N, int64_t K, int splits, int tps,
                   int rows_per_unit = BM) {
  GemmGeom g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.num_m = static_cast<int>(ceil_div(M, rows_per_unit));
  g.num_n = static_cast<int>(ceil_div(N, BN));
  g.num_kb = static_cast<int>(ceil_div(K, BK));
  g.splits = splits;
  g.tiles_per_split = tps;
  g.num_units = g.num_m * splits;
  g.timeout_ns = wait_timeout_ns();
  g.group_n = 0;
  return g;
}

int grid_for(const GemmGeom& g, int nsm) {
  return std::max(1, std::min(g.num_units, nsm));
}

// One contraction D[M,N] = A[M,K] B[K,N] as the kernels see it: each operand
// by its base pointer, row stride (elements) and major-ness.
struct GemmOperands {
  int64_t M, N, K;
  bool a_mn, b_mn;     // A stored [K][M] / B stored [K][N] (else [M][K], [N][K])
  const void* a;
  int64_t a_ld;
  const void* b;
  int64_t b_ld;
  bool sweep;          // sweep all column tiles per row block (choose splits)
  // B from two maps (GemmGeom::b_dual): 1 = along N (b2 has b's shape;
  // tiles of 128 output columns), 2 = along K (b covers k < k_split, b2
  // the rest; both have b's row stride)
  int b_dual = 0;
  const void* b2 = nullptr;
  int64_t k_split = 0;
};

struct GemmPlan {
  bool pair;
  GemmGeom g;
  CUtensorMap ta, tb, tb2;
  int grid;
};

lce_status plan_gemm(const GemmOperands& o, const DeviceInfo& dev,
                     GemmPlan* pl) {
  pl->pair = use_pair() && dev.pair_slots > 0;
  const int rows_unit = pl->pair ? 2 * BM : BM;
  const int slots = pl->pair ? dev.pair_slots : dev.num_sms;
  const int num_m = static_cast<int>(ceil_div(o.M, rows_unit));
  const int tile_n = o.b_dual == 1 ? BN / 2 : BN;
  const int num_n = static_cast<int>(ceil_div(o.N, tile_n));
  int splits = num_n, tps = 1;
  if (o.sweep) choose_splits(num_m, num_n, slots, o.K, &splits, &tps, rows_unit);
  pl->g = make_geom(o.M, o.N, o.K, splits, tps, rows_unit);
  pl->g.num_n = num_n;
  if (!o.sweep) pl->g.group_n = kGroupN;
  pl->g.b_dual = o.b_dual;
  pl->g.k_split_kb = o.b_dual == 2 ? static_cast<int>(o.k_split / BK) : 0;
  lce_status st = o.a_mn ? tmap_mnmajor(&pl->ta, o.a, o.M, o.K, o.a_ld)
                         : tmap_kmajor(&pl->ta, o.a, o.K, o.M, o.a_ld, BM);
  if (st != LCE_OK) return st;
  if (o.b_dual == 1) {  // K-major, 128-row boxes from each map
    st = tmap_kmajor(&pl->tb, o.b, o.K, o.N, o.b_ld, BM);
    if (st == LCE_OK) st = tmap_kmajor(&pl->tb2, o.b2, o.K, o.N, o.b_ld, BM);
  } else if (o.b_dual == 2) {  // MN-major, K split between the maps
    st = tmap_mnmajor(&pl->tb, o.b, o.N, o.k_split, o.b_ld);
    if (st == LCE_OK)
      st = tmap_mnmajor(&pl->tb2, o.b2, o.N, o.K - o.k_split, o.b_ld);
  } else {
    st = o.b_mn ? tmap_mnmajor(&pl->tb, o.b, o.N, o.K, o.b_ld)
                : tmap_kmajor(&pl->tb, o.b, o.K, o.N, o.b_ld,
                              pl->pair ? BM : BN);
    pl->tb2 = pl->tb;
  }
  if (st != LCE_OK) return st;
  const int units = std::max(1, std::min(pl->g.num_units, slots));
  pl->grid = pl->pair ? 2 * units : units;
  return LCE_OK;
}

// Turn on wave pacing for one launch: the counter is zeroed on the stream
// first. A wait runs out after ~two tiles' worth of MMA time at full rate.
cudaError_t pace(GemmPlan* pl, void* ctr, cudaStream_t s) {
  if (!wave_sync_on() || !ctr) return cudaSuccess;
  const GemmGeom& g = pl->g;
  const int slots = pl->pair ? pl->grid / 2 : pl->grid;
  // the most output tiles any CTA (cluster) walks, as the kernels assign
  // them (unit c, then every slots-th)
  uint32_t most = 0;
  for (int c = 0; c < slots; ++c) {
    uint32_t n = 0;
    for (int u = c; u < g.num_units; u += slots) {
      if (g.group_n > 0 && g.tiles_per_split == 1) {
        n += 1;
      } else {
        const int split = u % g.splits;
        n += static_cast<uint32_t>(
            std::min(g.tiles_per_split, g.num_n - split * g.tiles_per_split));
      }
    }
    most = std::max(most, n);
  }
  const double tile_flops = 2.0 * (pl->pair ? 2 * BM : BM) * BN * g.K;
  const double per_slot = 1.5e15 / (pl->pair ? 76 : 152);
  const double tile_ns = tile_flops / per_slot * 1e9;
  const double ns = 2.0 * tile_ns;
  pl->g.wave_ctr = static_cast<unsigned*>(ctr);
  pl->g.wave_wait_ns = static_cast<uint32_t>(
      std::min(2.0e6, std::max(2.0e4, ns)));
  pl->g.wave_steps = most;
  return cudaMemsetAsync(ctr, 0, sizeof(unsigned), s);
}

cudaError_t run_lse(const GemmPlan& pl, const LseParams& p, unsigned* err,
                    cudaStream_t s) {
  return pl.pair ? launch_gemm_pair_lse(pl.ta, pl.tb, pl.g, p, err, pl.grid, s)
                 : launch_gemm_lse(pl.ta, pl.tb, pl.g, p, err, pl.grid, s);
}
cudaError_t run_grad(const GemmPlan& pl, const GradParams& p,
                     const CUtensorMap& tg, unsigned* err, cudaStream_t s) {
  return pl.pair ? launch_gemm_pair_grad(pl.ta, pl.tb, tg, pl.g, p, err,
                                         pl.grid, s)
                 : launch_gemm_grad(pl.ta, pl.tb, tg, pl.g, p, err, pl.grid,
                                    s);
}
cudaError_t run_fused(const GemmPlan& pl, const FusedParams& p,
                      const CUtensorMap& te, unsigned* err, cudaStream_t s) {
  return pl.pair ? launch_gemm_pair_fused(pl.ta, pl.tb, te, pl.g, p, err,
                                          pl.grid, s)
                 : launch_gemm_fused(pl.ta, pl.tb, te, pl.g, p, err, pl.grid,
                                     s);
}
cudaError_t run_store(const GemmPlan& pl, bool a_mn, bool b_mn,
                      const StoreParams& p, unsigned* err, cudaStream_t s) {
  return pl.pair ? launch_gemm_pair_store(a_mn, b_mn, pl.ta, pl.tb, pl.g, p,
                                          err, pl.grid, s, &pl.tb2)
                 : launch_gemm_store(a_mn, b_mn, pl.ta, pl.tb, pl.g, p, err,
                                     pl.grid, s, &pl.tb2);
}

struct WsLayout {
  size_t n_valid, block_sums, part_m, part_s, part_z, zy, h16, w16, G,
      tile_max, total;
  size_t fwd_total;  // what the forward-only calls use: everything before G
  size_t sync;       // wave-pacing counter of the gradient contractions
  int64_t chunk, ldg;
};

bool sizes_ok(int64_t L, int64_t H, int64_t V) {
  return L >= 1 && H >= 8 && V >= 1 && H % 8 == 0 && L <= (1ll << 31) - BM &&
         V <= (1ll << 31) - BN && H <= (1ll << 31) - BK;
}

// Contraction slots and rows per work unit of the variant in use on the
// current device: CTA pairs (co-resident clusters, 256 rows) or single CTAs
// (SMs, 128 rows). Without a usable device, a GB300's values.
void slot_model(int* slots, int* rows_unit) {
  char saved[sizeof t_last_cuda_error];
  std::memcpy(saved, t_last_cuda_error, sizeof saved);
  DeviceInfo* dev = nullptr;
  const bool have = device_info(&dev) == LCE_OK;
  std::memcpy(t_last_cuda_error, saved, sizeof saved);
  const bool pair = use_pair() && (!have || dev->pair_slots > 0);
  *rows_unit = pair ? 2 * BM : BM;
  if (have)
    *slots = pair ? dev->pair_slots : dev->num_sms;
  else
    *slots = pair ? 76 : 152;
}

// Modelled time of one backward row chunk of cr rows, in units of one
// 64-deep k-slice of one output tile on one slot: the three contractions'
// waves times their k-slices, the dW read-add-write it adds (charged at a
// quarter of its DRAM time) and a fixed launch overhead (~0.1 ms).
double chunk_cost(int64_t cr, int64_t H, int64_t V, int slots, int rows_unit) {
  const double unit_s = 2.0 * rows_unit * BN * BK / 1.5e15 * slots;
  const int64_t nm = ceil_div(cr, rows_unit);
  const int64_t nh = ceil_div(H, BN);
  const int64_t nvn = ceil_div(V, BN), nvm = ceil_div(V, rows_unit);
  const double dh =
      static_cast<double>(ceil_div(nm * nh, slots)) * ceil_div(V, BK);
  int splits = 1, tps = static_cast<int>(nvn);
  choose_splits(static_cast<int>(nm), static_cast<int>(nvn), slots, H,
                &splits, &tps, rows_unit);
  const double lg = static_cast<double>(ceil_div(nm * splits, slots)) * tps *
                    ceil_div(H, BK);
  const double dw =
      static_cast<double>(ceil_div(nvm * nh, slots)) * ceil_div(cr, BK);
  const double rmw = (8.0 * V * H / 2.0e13) / unit_s;
  const double overhead = 1.0e-4 / unit_s;
  return dh + lg + dw + rmw + overhead;
}

// Row chunk of the backward when the caller passes 0: the multiple of 256
// rows, with the gradient-logit chunk within 8 GiB, that minimises the
// modelled time of all chunks (ties: the larger chunk).
int64_t default_chunk(int64_t L, int64_t H, int64_t V) {
  const double budget = 8.0 * (1ull << 30);
  const int64_t ldg = round_up(V, 8);
  const int64_t step = 2 * BM;
  int64_t cmax = static_cast<int64_t>(budget / (2.0 * ldg)) / step * step;
  cmax = std::max<int64_t>(cmax, step);
  cmax = std::min(cmax, round_up(L, step));
  int slots = 0, rows_unit = 0;
  slot_model(&slots, &rows_unit);
  int64_t best_c = cmax;
  double best = -1.0;
  for (int64_t c = cmax; c >= step; c -= step) {
    const int64_t full = L / c, rest = L - full * c;
    double cost = full * chunk_cost(c, H, V, slots, rows_unit);
    if (rest) cost += chunk_cost(rest, H, V, slots, rows_unit);
    if (best < 0 || cost < best * (1.0 - 1e-9)) {
      best = cost;
      best_c = c;
    }
  }
  return std::min(best_c, L);
}

WsLayout ws_layout(int64_t L, int64_t H, int64_t V, lce_dtype dt,
                   int64_t chunk_rows) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off + bytes), 256));
    return o;
  };
  w.chunk = chunk_rows > 0 ? std::min(chunk_rows, L) : default_chunk(L, H, V);
  w.ldg = round_up(V, 8);
  // per-256-row loss sums: one set over all rows (forward), or one set per
  // row chunk (fused forward+backward), whichever is longer
  const int64_t nchunks = ceil_div(L, w.chunk);
  const int64_t nb_fused = (nchunks - 1) * ceil_div(w.chunk, 256) +
                           ceil_div(L - (nchunks - 1) * w.chunk, 256);
  const int64_t nb = std::max(ceil_div(L, 256), nb_fused);
  w.n_valid = take(8);
  w.sync = take(8);
  w.block_sums = take(nb * 8);
  w.part_m = take(static_cast<size_t>(kMaxSplits) * L * 4);
  w.part_s = take(static_cast<size_t>(kMaxSplits) * L * 4);
  w.part_z = take(static_cast<size_t>(kMaxSplits) * L * 4);
  w.zy = take(L * 4);
  if (dt == LCE_F32) {
    w.h16 = take(static_cast<size_t>(L) * H * 2);
    w.w16 = take(static_cast<size_t>(V) * H * 2);
  } else {
    w.h16 = w.w16 = 0;
  }
  w.fwd_total = off;
  w.G = take(static_cast<size_t>(w.chunk) * w.ldg * 2);
  w.tile_max = take(static_cast<size_t>(w.chunk) * ceil_div(V, BN) * 4);
  w.total = off;
  return w;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Bring fp32 inputs to bf16 in the workspace; return the operand pointers.
lce_status operands(const void* h, const void* W, lce_dtype dt, int64_t L,
                    int64_t H, int64_t V, const WsLayout& w, uint8_t* ws,
                    cudaStream_t s, const void** hb, const void** Wb) {
  if (dt == LCE_BF16) {
    *hb = h;
    *Wb = W;
    return LCE_OK;
  }
  uint16_t* h16 = reinterpret_cast<uint16_t*>(ws + w.h16);
  uint16_t* w16 = reinterpret_cast<uint16_t*>(ws + w.w16);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_F32_TO_BF16, s);
    e = launch_f32_to_bf16(static_cast<const float*>(h), h16, L * H, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "f32_to_bf16(h)");
  {
    ProfScope ps(LCE_K_F32_TO_BF16, s);
    e = launch_f32_to_bf16(static_cast<const float*>(W), w16, V * H, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "f32_to_bf16(W)");
  *hb = h16;
  *Wb = w16;
  return LCE_OK;
}

// The loss variant of an optional lce_loss_opts: eps in [0, 1], zcoef >= 0
// with 2 zcoef finite (the gradient's factor); NULL is the plain loss.
struct Variant {
  float eps = 0.f, zcoef = 0.f;
  bool smooth() const { return eps != 0.f; }
  VariantGrad grad(int64_t V) const {
    VariantGrad v{2.f * zcoef, 1.f - eps, 0.f};
    if (eps != 0.f)
      v.eps_v = static_cast<float>(static_cast<double>(eps) /
                                   static_cast<double>(V));
    return v;
  }
};

bool read_variant(const lce_loss_opts* o, Variant* v) {
  *v = Variant{};
  if (!o) return true;
  if (!(o->label_smoothing >= 0.f && o->label_smoothing <= 1.f)) return false;
  if (!(o->z_loss >= 0.f) || !std::isfinite(2.f * o->z_loss)) return false;
  v->eps = o->label_smoothing;
  v->zcoef = o->z_loss;
  return true;
}

}  // namespace

// ---- scratch of lce_forward_static -----------------------------------------
// Callers that cannot allocate device memory (see lce_forward_static) get the
// forward's scratch from this fixed array instead of a caller workspace.
// Every GPU that loads the library holds these bytes until the process
// exits. Layout: the valid-row count, the per-block loss sums, the label
// logits, then the per-split (max, sum) partials.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int64_t kStaticMaxRows = 131072;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of g_static_scratch on the current device. The host-side
// name of the array is only a stand-in; the address is looked up once per
// device, with that device current, on the first lce_forward_static call.
lce_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_static_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LCE_OK;
}

}  // namespace
}  // namespace lce

using namespace lce;

extern "C" {

size_t lce_workspace_size(int64_t L, int64_t H, int64_t V, lce_dtype dt,
                          int64_t chunk_rows) {
  if (!sizes_ok(L, H, V) || chunk_rows < 0 || (dt != LCE_BF16 && dt != LCE_F32))
    return 0;
  return ws_layout(L, H, V, dt, chunk_rows).total;
}

int64_t lce_default_chunk_rows(int64_t L, int64_t H, int64_t V) {
  if (!sizes_ok(L, H, V)) return 0;
  return default_chunk(L, H, V);
}

lce_status lce_forward(const void* h, const void* W, lce_dtype dt,
                       const int64_t* labels, int64_t L, int64_t H, int64_t V,
                       int64_t ignore_index, float* loss, float* lse, void* ws,
                       size_t ws_bytes, void* stream) {
  return lce_forward_ex(h, W, dt, labels, L, H, V, ignore_index, nullptr, loss,
                        lse, ws, ws_bytes, stream);
}

lce_status lce_forward_ex(const void* h, const void* W, lce_dtype dt,
                          const int64_t* labels, int64_t L, int64_t H,
                          int64_t V, int64_t ignore_index,
                          const lce_loss_opts* opts, float* loss, float* lse,
                          void* ws, size_t ws_bytes, void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  if (!h || !W || !labels || !loss || !lse || !ws) return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, V)) return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u))
    return LCE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(L, H, V, dt, 0);
  if (ws_bytes < w.fwd_total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void *hb = nullptr, *Wb = nullptr;
  if ((st = operands(h, W, dt, L, H, V, w, wsb, s, &hb, &Wb)) != LCE_OK)
    return st;

  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb + w.n_valid);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V, ignore_index, n_valid, dev->err, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");

  // logits = h W^T: M = L rows, N = V columns, K = H
  GemmPlan pl;
  if ((st = plan_gemm({L, V, H, false, false, hb, H, Wb, H, true}, *dev,
                      &pl)) != LCE_OK)
    return st;
  const GemmGeom& g = pl.g;
  LseParams p{};
  p.labels = labels;
  p.part_m = reinterpret_cast<float*>(wsb + w.part_m);
  p.part_s = reinterpret_cast<float*>(wsb + w.part_s);
  p.zy = reinterpret_cast<float*>(wsb + w.zy);
  p.ignore_index = ignore_index;
  p.part_z = var.smooth() ? reinterpret_cast<float*>(wsb + w.part_z) : nullptr;
  e = pace(&pl, wsb + w.sync, s);
  if (e != cudaSuccess) return cuda_fail(e, "pace");
  {
    ProfScope ps(LCE_K_GEMM_LSE, s);
    e = run_lse(pl, p, dev->err, s);
    ps.done(2.0 * L * V * H);
  }
  if (e != cudaSuccess) return cuda_fail(e, "gemm_lse");

  int nblocks = 0;
  double* block_sums = reinterpret_cast<double*>(wsb + w.block_sums);
  {
    ProfScope ps(LCE_K_LSE_COMBINE, s);
    e = launch_lse_combine(p.part_m, p.part_s, g.splits, p.zy, labels, L, V,
                           ignore_index, lse, block_sums, &nblocks, s,
                           p.part_z, var.eps, var.zcoef);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "lse_combine");
  {
    ProfScope ps(LCE_K_LOSS_FINALIZE, s);
    e = launch_loss_finalize(block_sums, nblocks, n_valid, loss, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "loss_finalize");
  return LCE_OK;
}

}  // extern "C"

namespace lce {
namespace {

// The backward over the vocabulary columns [v0, v0 + V) of a vocabulary of
// V_total (lce_backward: v0 = 0, V_total = V); dH in dt, or in fp32 when
// dh_f32.
lce_status backward_impl(const void* h, const void* W, lce_dtype dt,
                         const int64_t* labels, const float* lse, int64_t L,
                         int64_t H, int64_t V, int64_t v0, int64_t V_total,
                         int64_t ignore_index, const float* dloss,
                         int64_t chunk_rows, void* dH, bool dh_f32, float* dW,
                         void* ws, size_t ws_bytes, void* stream,
                         const VariantGrad& var) {
  // dH or dW may be NULL (that gradient is not computed), not both
  if (!h || !W || !labels || !lse || !dloss || (!dH && !dW) || !ws)
    return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, V) || chunk_rows < 0) return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) || !aligned16(dH) ||
      !aligned16(dW) || (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(dloss) & 3u))
    return LCE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(L, H, V, dt, chunk_rows);
  if (ws_bytes < w.total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void *hb = nullptr, *Wb = nullptr;
  if ((st = operands(h, W, dt, L, H, V, w, wsb, s, &hb, &Wb)) != LCE_OK)
    return st;

  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb + w.n_valid);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V_total, ignore_index, n_valid, dev->err,
                           s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");

  uint16_t* G = reinterpret_cast<uint16_t*>(wsb + w.G);
  const size_t dh_elem = (dh_f32 || dt == LCE_F32) ? 4 : 2;

  for (int64_t c0 = 0; c0 < L; c0 += w.chunk) {
    const int64_t cr = std::min(w.chunk, L - c0);
    const uint16_t* hc = static_cast<const uint16_t*>(hb) + c0 * H;

    // (1) recompute z_c = h_c W^T and write G_c = softmax - onehot (bf16)
    {
      GemmPlan pl;
      if ((st = plan_gemm({cr, V, H, false, false, hc, H, Wb, H, true},
                          *dev, &pl)) != LCE_OK)
        return st;
      GradParams p{};
      p.labels = labels + c0;
      p.lse = lse + c0;
      p.G = G;
      p.ldg = w.ldg;
      p.ignore_index = ignore_index;
      p.v0 = v0;
      p.v_total = V_total;
      p.var = var;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      CUtensorMap tg;
      if ((st = tmap_store_box(&tg, G, V, cr, w.ldg)) != LCE_OK) return st;
      ProfScope ps(LCE_K_GEMM_GRAD, s);
      e = run_grad(pl, p, tg, dev->err, s);
      ps.done(2.0 * cr * V * H);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_grad");
    }
    // (2) dH_c = (dloss/N) G_c W: M = cr, N = H, K = V
    if (dH) {
      GemmPlan pl;
      if ((st = plan_gemm({cr, H, V, false, true, G, w.ldg, Wb, H, false},
                          *dev, &pl)) != LCE_OK)
        return st;
      StoreParams p{};
      p.out = static_cast<uint8_t*>(dH) + c0 * H * dh_elem;
      p.ldo = H;
      p.out_f32 = dh_f32 || dt == LCE_F32;
      p.accumulate = 0;
      p.dloss = dloss;
      p.n_valid = n_valid;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      ProfScope ps(LCE_K_GEMM_DH, s);
      e = run_store(pl, false, true, p, dev->err, s);
      ps.done(2.0 * cr * H * V);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_dH");
    }
    // (3) dW (+)= (dloss/N) G_c^T h_c: M = V, N = H, K = cr
    if (dW) {
      GemmPlan pl;
      if ((st = plan_gemm({V, H, cr, true, true, G, w.ldg, hc, H, false},
                          *dev, &pl)) != LCE_OK)
        return st;
      StoreParams p{};
      p.out = dW;
      p.ldo = H;
      p.out_f32 = 1;
      p.accumulate = c0 > 0;
      p.dloss = dloss;
      p.n_valid = n_valid;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      ProfScope ps(LCE_K_GEMM_DW, s);
      e = run_store(pl, true, true, p, dev->err, s);
      ps.done(2.0 * V * H * cr);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_dW");
    }
  }
  return LCE_OK;
}

}  // namespace
}  // namespace lce

extern "C" {

lce_status lce_backward(const void* h, const void* W, lce_dtype dt,
                        const int64_t* labels, const float* lse, int64_t L,
                        int64_t H, int64_t V, int64_t ignore_index,
                        const float* dloss, int64_t chunk_rows, void* dH,
                        float* dW, void* ws, size_t ws_bytes, void* stream) {
  return lce_backward_ex(h, W, dt, labels, lse, L, H, V, ignore_index,
                         nullptr, dloss, chunk_rows, dH, dW, ws, ws_bytes,
                         stream);
}

lce_status lce_backward_ex(const void* h, const void* W, lce_dtype dt,
                           const int64_t* labels, const float* lse, int64_t L,
                           int64_t H, int64_t V, int64_t ignore_index,
                           const lce_loss_opts* opts, const float* dloss,
                           int64_t chunk_rows, void* dH, float* dW, void* ws,
                           size_t ws_bytes, void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  return backward_impl(h, W, dt, labels, lse, L, H, V, 0, V, ignore_index,
                       dloss, chunk_rows, dH, false, dW, ws, ws_bytes, stream,
                       var.grad(V));
}

lce_status lce_backward_slice(const void* h, const void* W, lce_dtype dt,
                              const int64_t* labels, const float* lse,
                              int64_t L, int64_t H, int64_t Vs, int64_t v0,
                              int64_t V_total, int64_t ignore_index,
                              const float* dloss, int64_t chunk_rows,
                              float* dH_part, float* dW, void* ws,
                              size_t ws_bytes, void* stream) {
  return lce_backward_slice_ex(h, W, dt, labels, lse, L, H, Vs, v0, V_total,
                               ignore_index, nullptr, dloss, chunk_rows,
                               dH_part, dW, ws, ws_bytes, stream);
}

lce_status lce_backward_slice_ex(const void* h, const void* W, lce_dtype dt,
                                 const int64_t* labels, const float* lse,
                                 int64_t L, int64_t H, int64_t Vs, int64_t v0,
                                 int64_t V_total, int64_t ignore_index,
                                 const lce_loss_opts* opts,
                                 const float* dloss, int64_t chunk_rows,
                                 float* dH_part, float* dW, void* ws,
                                 size_t ws_bytes, void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  if (v0 < 0 || Vs < 1 || V_total < 1 || v0 > V_total - Vs)
    return LCE_ERR_INVALID_ARG;
  return backward_impl(h, W, dt, labels, lse, L, H, Vs, v0, V_total,
                       ignore_index, dloss, chunk_rows, dH_part, true, dW, ws,
                       ws_bytes, stream, var.grad(V_total));
}

}  // extern "C"

namespace lce {
namespace {

// One vocabulary slice's forward statistics: the logits pass with the
// statistics epilogue, or (keep_exp) with the fused epilogue that also keeps
// the slice's tile exponentials in ws; then the split partials merged into
// m, s, zy and, when zsum is given, the slice's logit sums.
lce_status forward_slice_impl(bool keep_exp, const void* h, const void* W,
                              lce_dtype dt, const int64_t* labels, int64_t L,
                              int64_t H, int64_t Vs, int64_t v0,
                              int64_t V_total, int64_t ignore_index,
                              const lce_loss_opts* opts, float* m,
                              float* s_out, float* zy, float* zsum, void* ws,
                              size_t ws_bytes, void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  if (!h || !W || !labels || !m || !s_out || !zy || !ws)
    return LCE_ERR_INVALID_ARG;
  if (var.smooth() && !zsum) return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, Vs) || v0 < 0 || V_total < 1 || v0 > V_total - Vs)
    return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(m) & 3u) ||
      (reinterpret_cast<uintptr_t>(s_out) & 3u) ||
      (reinterpret_cast<uintptr_t>(zy) & 3u) ||
      (reinterpret_cast<uintptr_t>(zsum) & 3u))
    return LCE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(L, H, Vs, dt, keep_exp ? L : 0);
  if (ws_bytes < (keep_exp ? w.total : w.fwd_total)) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void *hb = nullptr, *Wb = nullptr;
  if ((st = operands(h, W, dt, L, H, Vs, w, wsb, s, &hb, &Wb)) != LCE_OK)
    return st;
  // the label range check against the whole vocabulary
  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb + w.n_valid);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V_total, ignore_index, n_valid,
                           dev->err, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");
  GemmPlan pl;
  if ((st = plan_gemm({L, Vs, H, false, false, hb, H, Wb, H, true},
                      *dev, &pl)) != LCE_OK)
    return st;
  float* part_m = reinterpret_cast<float*>(wsb + w.part_m);
  float* part_s = reinterpret_cast<float*>(wsb + w.part_s);
  float* zy_in = reinterpret_cast<float*>(wsb + w.zy);
  float* part_z = zsum ? reinterpret_cast<float*>(wsb + w.part_z) : nullptr;
  e = pace(&pl, wsb + w.sync, s);
  if (e != cudaSuccess) return cuda_fail(e, "pace");
  if (keep_exp) {
    // every row's logits once: statistics + tile exponentials kept in ws
    uint16_t* E = reinterpret_cast<uint16_t*>(wsb + w.G);
    FusedParams p{};
    p.labels = labels;
    p.part_m = part_m;
    p.part_s = part_s;
    p.zy = zy_in;
    p.part_z = part_z;
    p.E = E;
    p.ldg = w.ldg;
    p.tile_max = reinterpret_cast<float*>(wsb + w.tile_max);
    p.ignore_index = ignore_index;
    p.v0 = v0;
    p.v_total = V_total;
    CUtensorMap te;
    if ((st = tmap_store_box(&te, E, Vs, L, w.ldg)) != LCE_OK) return st;
    ProfScope ps(LCE_K_GEMM_FUSED, s);
    e = run_fused(pl, p, te, dev->err, s);
    ps.done(2.0 * L * Vs * H);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_fused");
  } else {
    LseParams p{};
    p.labels = labels;
    p.part_m = part_m;
    p.part_s = part_s;
    p.zy = zy_in;
    p.part_z = part_z;
    p.ignore_index = ignore_index;
    p.v0 = v0;
    p.v_total = V_total;
    ProfScope ps(LCE_K_GEMM_LSE, s);
    e = run_lse(pl, p, dev->err, s);
    ps.done(2.0 * L * Vs * H);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_lse");
  }
  {
    ProfScope ps(LCE_K_SLICE_STATS, s);
    e = launch_slice_stats(part_m, part_s, pl.g.splits, zy_in, labels, L, v0,
                           Vs, V_total, ignore_index, m, s_out, zy, s, part_z,
                           zsum);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "slice_stats");
  return LCE_OK;
}

}  // namespace
}  // namespace lce

extern "C" {

lce_status lce_forward_slice(const void* h, const void* W, lce_dtype dt,
                             const int64_t* labels, int64_t L, int64_t H,
                             int64_t Vs, int64_t v0, int64_t V_total,
                             int64_t ignore_index, float* m, float* s_out,
                             float* zy, void* ws, size_t ws_bytes,
                             void* stream) {
  return forward_slice_impl(false, h, W, dt, labels, L, H, Vs, v0, V_total,
                            ignore_index, nullptr, m, s_out, zy, nullptr, ws,
                            ws_bytes, stream);
}

lce_status lce_forward_slice_ex(const void* h, const void* W, lce_dtype dt,
                                const int64_t* labels, int64_t L, int64_t H,
                                int64_t Vs, int64_t v0, int64_t V_total,
                                int64_t ignore_index,
                                const lce_loss_opts* opts, float* m,
                                float* s_out, float* zy, float* zsum,
                                void* ws, size_t ws_bytes, void* stream) {
  return forward_slice_impl(false, h, W, dt, labels, L, H, Vs, v0, V_total,
                            ignore_index, opts, m, s_out, zy, zsum, ws,
                            ws_bytes, stream);
}

size_t lce_slice_exp_workspace_size(int64_t L, int64_t H, int64_t Vs,
                                    lce_dtype dt) {
  if (!sizes_ok(L, H, Vs) || (dt != LCE_BF16 && dt != LCE_F32)) return 0;
  return ws_layout(L, H, Vs, dt, L).total;
}

lce_status lce_forward_slice_exp(const void* h, const void* W, lce_dtype dt,
                                 const int64_t* labels, int64_t L, int64_t H,
                                 int64_t Vs, int64_t v0, int64_t V_total,
                                 int64_t ignore_index, float* m, float* s_out,
                                 float* zy, void* ws, size_t ws_bytes,
                                 void* stream) {
  return forward_slice_impl(true, h, W, dt, labels, L, H, Vs, v0, V_total,
                            ignore_index, nullptr, m, s_out, zy, nullptr, ws,
                            ws_bytes, stream);
}

lce_status lce_forward_slice_exp_ex(const void* h, const void* W,
                                    lce_dtype dt, const int64_t* labels,
                                    int64_t L, int64_t H, int64_t Vs,
                                    int64_t v0, int64_t V_total,
                                    int64_t ignore_index,
                                    const lce_loss_opts* opts, float* m,
                                    float* s_out, float* zy, float* zsum,
                                    void* ws, size_t ws_bytes, void* stream) {
  return forward_slice_impl(true, h, W, dt, labels, L, H, Vs, v0, V_total,
                            ignore_index, opts, m, s_out, zy, zsum, ws,
                            ws_bytes, stream);
}

lce_status lce_backward_slice_exp(const void* h, const void* W, lce_dtype dt,
                                  const int64_t* labels, const float* lse,
                                  int64_t L, int64_t H, int64_t Vs, int64_t v0,
                                  int64_t V_total, int64_t ignore_index,
                                  const float* dloss, float* dH_part,
                                  float* dW, void* ws, size_t ws_bytes,
                                  void* stream) {
  return lce_backward_slice_exp_ex(h, W, dt, labels, lse, L, H, Vs, v0,
                                   V_total, ignore_index, nullptr, dloss,
                                   dH_part, dW, ws, ws_bytes, stream);
}

lce_status lce_backward_slice_exp_ex(const void* h, const void* W,
                                     lce_dtype dt, const int64_t* labels,
                                     const float* lse, int64_t L, int64_t H,
                                     int64_t Vs, int64_t v0, int64_t V_total,
                                     int64_t ignore_index,
                                     const lce_loss_opts* opts,
                                     const float* dloss, float* dH_part,
                                     float* dW, void* ws, size_t ws_bytes,
                                     void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  // dH_part or dW may be NULL (not computed), not both
  if (!h || !W || !labels || !lse || !dloss || (!dH_part && !dW) || !ws)
    return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, Vs) || v0 < 0 || V_total < 1 || v0 > V_total - Vs)
    return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) ||
      !aligned16(dH_part) || !aligned16(dW) ||
      (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(dloss) & 3u))
    return LCE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(L, H, Vs, dt, L);
  if (ws_bytes < w.total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void *hb = nullptr, *Wb = nullptr;
  if ((st = operands(h, W, dt, L, H, Vs, w, wsb, s, &hb, &Wb)) != LCE_OK)
    return st;
  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb + w.n_valid);
  uint16_t* E = reinterpret_cast<uint16_t*>(wsb + w.G);
  const int num_n = static_cast<int>(ceil_div(Vs, BN));
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V_total, ignore_index, n_valid,
                           dev->err, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");
  // the kept exponentials -> softmax - onehot with the merged lse
  {
    ProfScope ps(LCE_K_GRAD_FROM_EXP, s);
    e = launch_grad_from_exp(E, w.ldg,
                             reinterpret_cast<float*>(wsb + w.tile_max), num_n,
                             lse, labels, L, Vs, ignore_index, dev->num_sms, s,
                             v0, V_total, var.grad(V_total));
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "grad_from_exp");
  // dH_part = (dloss/N) G W_s: M = L, N = H, K = Vs
  if (dH_part) {
    GemmPlan pl;
    if ((st = plan_gemm({L, H, Vs, false, true, E, w.ldg, Wb, H, false},
                        *dev, &pl)) != LCE_OK)
      return st;
    StoreParams p{};
    p.out = dH_part;
    p.ldo = H;
    p.out_f32 = 1;
    p.accumulate = 0;
    p.dloss = dloss;
    p.n_valid = n_valid;
    e = pace(&pl, wsb + w.sync, s);
    if (e != cudaSuccess) return cuda_fail(e, "pace");
    ProfScope ps(LCE_K_GEMM_DH, s);
    e = run_store(pl, false, true, p, dev->err, s);
    ps.done(2.0 * L * H * Vs);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_dH");
  }
  // dW_s = (dloss/N) G^T h: M = Vs, N = H, K = L, written once
  if (dW) {
    GemmPlan pl;
    if ((st = plan_gemm({Vs, H, L, true, true, E, w.ldg, hb, H, false},
                        *dev, &pl)) != LCE_OK)
      return st;
    StoreParams p{};
    p.out = dW;
    p.ldo = H;
    p.out_f32 = 1;
    p.accumulate = 0;
    p.dloss = dloss;
    p.n_valid = n_valid;
    e = pace(&pl, wsb + w.sync, s);
    if (e != cudaSuccess) return cuda_fail(e, "pace");
    ProfScope ps(LCE_K_GEMM_DW, s);
    e = run_store(pl, true, true, p, dev->err, s);
    ps.done(2.0 * Vs * H * L);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_dW");
  }
  return LCE_OK;
}

size_t lce_combine_workspace_size(int64_t L) {
  if (L < 1) return 0;
  return 256 + static_cast<size_t>(ceil_div(L, COMBINE_ROWS)) * 8;
}

lce_status lce_combine_slices(const float* m, const float* s_in,
                              const float* zy, int64_t P,
                              const int64_t* labels, int64_t L,
                              int64_t V_total, int64_t ignore_index,
                              float* loss, float* lse, void* ws,
                              size_t ws_bytes, void* stream) {
  return lce_combine_slices_ex(m, s_in, zy, nullptr, P, labels, L, V_total,
                               ignore_index, nullptr, loss, lse, ws, ws_bytes,
                               stream);
}

lce_status lce_combine_slices_ex(const float* m, const float* s_in,
                                 const float* zy, const float* zsum, int64_t P,
                                 const int64_t* labels, int64_t L,
                                 int64_t V_total, int64_t ignore_index,
                                 const lce_loss_opts* opts, float* loss,
                                 float* lse, void* ws, size_t ws_bytes,
                                 void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  if (!m || !s_in || !zy || !labels || !loss || !lse || !ws || P < 1 ||
      L < 1 || V_total < 1)
    return LCE_ERR_INVALID_ARG;
  if (var.smooth() && !zsum) return LCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(m) & 3u) ||
      (reinterpret_cast<uintptr_t>(s_in) & 3u) ||
      (reinterpret_cast<uintptr_t>(zy) & 3u) ||
      (reinterpret_cast<uintptr_t>(zsum) & 3u) ||
      (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || !aligned16(ws))
    return LCE_ERR_INVALID_ARG;
  if (ws_bytes < lce_combine_workspace_size(L)) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb);
  double* block_sums = reinterpret_cast<double*>(wsb + 256);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V_total, ignore_index, n_valid,
                           dev->err, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");
  int nb = 0;
  {
    ProfScope ps(LCE_K_COMBINE_SLICES, s);
    // the logit sums only enter under label smoothing: without it the
    // terms are the plain loss's, bit for bit, whatever zsum holds
    e = launch_combine_slices(m, s_in, zy, P, labels, L, V_total, ignore_index,
                              lse, block_sums, &nb, s,
                              var.smooth() ? zsum : nullptr, var.eps,
                              var.zcoef);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "combine_slices");
  {
    ProfScope ps(LCE_K_LOSS_FINALIZE, s);
    e = launch_loss_finalize(block_sums, nb, n_valid, loss, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "loss_finalize");
  return LCE_OK;
}

lce_status lce_forward_backward(const void* h, const void* W, lce_dtype dt,
                                const int64_t* labels, int64_t L, int64_t H,
                                int64_t V, int64_t ignore_index,
                                int64_t chunk_rows, float* loss, float* lse,
                                void* dH, float* dW, void* ws, size_t ws_bytes,
                                void* stream) {
  return lce_forward_backward_ex(h, W, dt, labels, L, H, V, ignore_index,
                                 nullptr, chunk_rows, loss, lse, dH, dW, ws,
                                 ws_bytes, stream);
}

lce_status lce_forward_backward_ex(const void* h, const void* W, lce_dtype dt,
                                   const int64_t* labels, int64_t L, int64_t H,
                                   int64_t V, int64_t ignore_index,
                                   const lce_loss_opts* opts,
                                   int64_t chunk_rows, float* loss, float* lse,
                                   void* dH, float* dW, void* ws,
                                   size_t ws_bytes, void* stream) {
  Variant var;
  if (!read_variant(opts, &var)) return LCE_ERR_INVALID_ARG;
  const VariantGrad vg = var.grad(V);
  // dH and dW may each be NULL: that gradient is not computed
  if (!h || !W || !labels || !loss || !lse || !ws) return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, V) || chunk_rows < 0) return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws) || !aligned16(dH) ||
      !aligned16(dW) || (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u))
    return LCE_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(L, H, V, dt, chunk_rows);
  if (ws_bytes < w.total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void *hb = nullptr, *Wb = nullptr;
  if ((st = operands(h, W, dt, L, H, V, w, wsb, s, &hb, &Wb)) != LCE_OK)
    return st;

  auto* n_valid = reinterpret_cast<unsigned long long*>(wsb + w.n_valid);
  cudaError_t e;
  {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V, ignore_index, n_valid, dev->err, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");

  uint16_t* E = reinterpret_cast<uint16_t*>(wsb + w.G);
  float* tile_max = reinterpret_cast<float*>(wsb + w.tile_max);
  float* part_m = reinterpret_cast<float*>(wsb + w.part_m);
  float* part_s = reinterpret_cast<float*>(wsb + w.part_s);
  float* part_z =
      var.smooth() ? reinterpret_cast<float*>(wsb + w.part_z) : nullptr;
  float* zy = reinterpret_cast<float*>(wsb + w.zy);
  double* block_sums = reinterpret_cast<double*>(wsb + w.block_sums);
  const size_t dh_elem = dt == LCE_F32 ? 4 : 2;
  const int num_n = static_cast<int>(ceil_div(V, BN));

  int block_off = 0;
  for (int64_t c0 = 0; c0 < L; c0 += w.chunk) {
    const int64_t cr = std::min(w.chunk, L - c0);
    const uint16_t* hc = static_cast<const uint16_t*>(hb) + c0 * H;
    // (1) logits of the chunk -> forward statistics + tile exponentials
    int splits = 1;
    {
      GemmPlan pl;
      if ((st = plan_gemm({cr, V, H, false, false, hc, H, Wb, H, true},
                          *dev, &pl)) != LCE_OK)
        return st;
      splits = pl.g.splits;
      FusedParams p{};
      p.labels = labels + c0;
      p.part_m = part_m;
      p.part_s = part_s;
      p.zy = zy;
      p.E = E;
      p.ldg = w.ldg;
      p.tile_max = tile_max;
      p.ignore_index = ignore_index;
      p.part_z = part_z;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      CUtensorMap te;
      if ((st = tmap_store_box(&te, E, V, cr, w.ldg)) != LCE_OK) return st;
      ProfScope ps(LCE_K_GEMM_FUSED, s);
      e = run_fused(pl, p, te, dev->err, s);
      ps.done(2.0 * cr * V * H);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_fused");
    }
    // (2) the chunk's lse and loss terms
    {
      int nb = 0;
      ProfScope ps(LCE_K_LSE_COMBINE, s);
      e = launch_lse_combine(part_m, part_s, splits, zy, labels + c0, cr, V,
                             ignore_index, lse + c0, block_sums + block_off,
                             &nb, s, part_z, var.eps, var.zcoef);
      ps.done(0);
      if (e != cudaSuccess) return cuda_fail(e, "lse_combine");
      block_off += nb;
    }
    // (3) exponentials -> softmax - onehot, in place
    if (dH || dW) {
      ProfScope ps(LCE_K_GRAD_FROM_EXP, s);
      e = launch_grad_from_exp(E, w.ldg, tile_max, num_n, lse + c0,
                               labels + c0, cr, V, ignore_index, dev->num_sms,
                               s, 0, 0, vg);
      ps.done(0);
      if (e != cudaSuccess) return cuda_fail(e, "grad_from_exp");
    }
    // (4) dH_c = G_c W / N
    if (dH) {
      GemmPlan pl;
      if ((st = plan_gemm({cr, H, V, false, true, E, w.ldg, Wb, H, false},
                          *dev, &pl)) != LCE_OK)
        return st;
      StoreParams p{};
      p.out = static_cast<uint8_t*>(dH) + c0 * H * dh_elem;
      p.ldo = H;
      p.out_f32 = dt == LCE_F32;
      p.accumulate = 0;
      p.dloss = nullptr;
      p.n_valid = n_valid;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      ProfScope ps(LCE_K_GEMM_DH, s);
      e = run_store(pl, false, true, p, dev->err, s);
      ps.done(2.0 * cr * H * V);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_dH");
    }
    // (5) dW (+)= G_c^T h_c / N
    if (dW) {
      GemmPlan pl;
      if ((st = plan_gemm({V, H, cr, true, true, E, w.ldg, hc, H, false},
                          *dev, &pl)) != LCE_OK)
        return st;
      StoreParams p{};
      p.out = dW;
      p.ldo = H;
      p.out_f32 = 1;
      p.accumulate = c0 > 0;
      p.dloss = nullptr;
      p.n_valid = n_valid;
      e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      ProfScope ps(LCE_K_GEMM_DW, s);
      e = run_store(pl, true, true, p, dev->err, s);
      ps.done(2.0 * V * H * cr);
      if (e != cudaSuccess) return cuda_fail(e, "gemm_dW");
    }
  }
  {
    ProfScope ps(LCE_K_LOSS_FINALIZE, s);
    e = launch_loss_finalize(block_sums, block_off, n_valid, loss, s);
    ps.done(0);
  }
  if (e != cudaSuccess) return cuda_fail(e, "loss_finalize");
  return LCE_OK;
}

lce_status lce_scale_gradients(void* dH, lce_dtype dt, int64_t L, int64_t H,
                               float* dW, int64_t V, const float* dloss,
                               void* stream) {
  // either gradient may be NULL (not scaled)
  if (!dloss) return LCE_ERR_INVALID_ARG;
  if (dt != LCE_BF16 && dt != LCE_F32) return LCE_ERR_UNSUPPORTED;
  if (!sizes_ok(L, H, V)) return LCE_ERR_INVALID_ARG;
  if (!aligned16(dH) || !aligned16(dW) ||
      (reinterpret_cast<uintptr_t>(dloss) & 3u))
    return LCE_ERR_INVALID_ARG;
  if (!dH && !dW) return LCE_OK;  // nothing to scale
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(LCE_K_SCALE_GRADS, s);
  cudaError_t e = launch_scale_grads(dH, dt == LCE_F32, dH ? L * H : 0, dW,
                                     dW ? V * H : 0, dloss, s);
  ps.done(0);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "scale_grads");
}

lce_status lce_count_valid(const int64_t* labels, int64_t L, int64_t V,
                           int64_t ignore_index, int64_t* n_valid,
                           void* stream) {
  if (!n_valid || (L > 0 && !labels) || L < 0 || V < 1) return LCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(n_valid) & 7u))
    return LCE_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* n = reinterpret_cast<unsigned long long*>(n_valid);
  cudaError_t e;
  if (L == 0) {
    e = cudaMemsetAsync(n, 0, sizeof(unsigned long long), s);
  } else {
    ProfScope ps(LCE_K_COUNT_VALID, s);
    e = launch_count_valid(labels, L, V, ignore_index, n, dev->err, s);
    ps.done(0);
  }
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "count_valid");
}

lce_status lce_shard_sums(const float* loss_local, const int64_t* n_local,
                          double* sums, void* stream) {
  if (!loss_local || !n_local || !sums) return LCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(loss_local) & 3u) ||
      (reinterpret_cast<uintptr_t>(n_local) & 7u) ||
      (reinterpret_cast<uintptr_t>(sums) & 7u))
    return LCE_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(LCE_K_SHARD_COMBINE, s);
  cudaError_t e = launch_shard_sums(
      loss_local, reinterpret_cast<const unsigned long long*>(n_local), sums,
      s);
  ps.done(0);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "shard_sums");
}

lce_status lce_combine_shards(const double* sums, const int64_t* n_local,
                              const float* dloss, float* loss, float* weight,
                              void* stream) {
  if (!sums || !n_local || !loss || !weight) return LCE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(sums) & 7u) ||
      (reinterpret_cast<uintptr_t>(n_local) & 7u) ||
      (reinterpret_cast<uintptr_t>(dloss) & 3u) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u) ||
      (reinterpret_cast<uintptr_t>(weight) & 3u))
    return LCE_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(LCE_K_SHARD_COMBINE, s);
  cudaError_t e = launch_combine_shards(
      sums, reinterpret_cast<const unsigned long long*>(n_local), dloss, loss,
      weight, s);
  ps.done(0);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "combine_shards");
}

// ---- sequence-tiled gated MLP ----------------------------------------------

}  // extern "C"

namespace lce {
namespace {

struct MlpLayout {
  size_t sync, g, u, a, dgu, total;
  int64_t chunk;
};

bool mlp_sizes_ok(int64_t L, int64_t H, int64_t I) {
  return L >= 1 && H >= 8 && I >= 64 && H % 8 == 0 && I % 64 == 0 &&
         L <= (1ll << 31) - 2 * BM && H <= (1ll << 30) && I <= (1ll << 29);
}

// Row chunk of the MLP: the chunk's four intermediates (g, u, a and
// [dg | du], 10 I bytes per row) within 4 GiB, in multiples of 256 rows,
// split evenly.
int64_t mlp_default_chunk(int64_t L, int64_t I) {
  const double budget = 4.0 * (1ull << 30);
  const int64_t step = 2 * BM;
  int64_t cmax = static_cast<int64_t>(budget / (10.0 * I)) / step * step;
  cmax = std::max<int64_t>(cmax, step);
  const int64_t n = ceil_div(L, cmax);
  return std::min(round_up(ceil_div(L, n), step), L);
}

MlpLayout mlp_layout(int64_t L, int64_t I, int64_t chunk_rows) {
  MlpLayout w{};
  w.chunk = chunk_rows > 0 ? std::min(chunk_rows, L) : mlp_default_chunk(L, I);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off + bytes), 256));
    return o;
  };
  const size_t plane = static_cast<size_t>(w.chunk) * I * 2;
  w.sync = take(8);
  w.g = take(plane);
  w.u = take(plane);
  w.a = take(plane);
  w.dgu = take(2 * plane);
  w.total = off;
  return w;
}

// a_c = silu(x_c Wg^T) * (x_c Wu^T), optionally saving g_c and u_c.
lce_status mlp_gate_up(const DeviceInfo& dev, const uint16_t* xc, int64_t cr,
                       const void* Wg, const void* Wu, int64_t H, int64_t I,
                       uint16_t* a, uint16_t* g, uint16_t* u, void* ctr,
                       cudaStream_t s) {
  GemmOperands o{cr, I, H, false, false, xc, H, Wg, H, false};
  o.b_dual = 1;
  o.b2 = Wu;
  GemmPlan pl;
  lce_status st = plan_gemm(o, dev, &pl);
  if (st != LCE_OK) return st;
  SwigluParams p{};
  if ((st = tmap_store_box(&p.map_a, a, I, cr, I)) != LCE_OK) return st;
  p.save_gu = g != nullptr && u != nullptr;
  if (p.save_gu) {
    if ((st = tmap_store_box(&p.map_g, g, I, cr, I)) != LCE_OK) return st;
    if ((st = tmap_store_box(&p.map_u, u, I, cr, I)) != LCE_OK) return st;
  }
  cudaError_t e = pace(&pl, ctr, s);
  if (e != cudaSuccess) return cuda_fail(e, "pace");
  ProfScope ps(LCE_K_MLP_GATE_UP, s);
  e = launch_gemm_swiglu(pl.pair, pl.ta, pl.tb, pl.tb2, pl.g, p, dev.err,
                         pl.grid, s);
  ps.done(2.0 * cr * H * 2 * I);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "mlp_gate_up");
}

// out (+)= scale * (A B) for the plain MLP contractions.
lce_status mlp_store(const DeviceInfo& dev, const GemmOperands& o,
                     const StoreParams& p, int kind, void* ctr,
                     cudaStream_t s) {
  GemmPlan pl;
  lce_status st = plan_gemm(o, dev, &pl);
  if (st != LCE_OK) return st;
  cudaError_t e = pace(&pl, ctr, s);
  if (e != cudaSuccess) return cuda_fail(e, "pace");
  ProfScope ps(kind, s);
  e = run_store(pl, o.a_mn, o.b_mn, p, dev.err, s);
  ps.done(2.0 * o.M * o.N * o.K);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "mlp contraction");
}

lce_status mlp_check(const void* x, const void* Wg, const void* Wu,
                     const void* Wd, int64_t L, int64_t H, int64_t I) {
  if (!x || !Wg || !Wu || !Wd) return LCE_ERR_INVALID_ARG;
  if (!mlp_sizes_ok(L, H, I)) return LCE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd))
    return LCE_ERR_INVALID_ARG;
  return LCE_OK;
}

}  // namespace
}  // namespace lce

extern "C" {

size_t lce_mlp_workspace_size(int64_t L, int64_t H, int64_t I,
                              int64_t chunk_rows) {
  if (!mlp_sizes_ok(L, H, I) || chunk_rows < 0) return 0;
  return mlp_layout(L, I, chunk_rows).total;
}

lce_status lce_mlp_forward(const void* x, const void* Wg, const void* Wu,
                           const void* Wd, int64_t L, int64_t H, int64_t I,
                           int64_t chunk_rows, void* y, void* ws,
                           size_t ws_bytes, void* stream) {
  lce_status st = mlp_check(x, Wg, Wu, Wd, L, H, I);
  if (st != LCE_OK) return st;
  if (!y || !ws || !aligned16(y) || !aligned16(ws) || chunk_rows < 0)
    return LCE_ERR_INVALID_ARG;
  const MlpLayout w = mlp_layout(L, I, chunk_rows);
  if (ws_bytes < w.total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint16_t* A = reinterpret_cast<uint16_t*>(wsb + w.a);
  for (int64_t c0 = 0; c0 < L; c0 += w.chunk) {
    const int64_t cr = std::min(w.chunk, L - c0);
    const uint16_t* xc = static_cast<const uint16_t*>(x) + c0 * H;
    // a_c = silu(x_c Wg^T) * (x_c Wu^T)
    if ((st = mlp_gate_up(*dev, xc, cr, Wg, Wu, H, I, A, nullptr, nullptr,
                          wsb + w.sync, s)) != LCE_OK)
      return st;
    // y_c = a_c Wd^T
    StoreParams p{};
    p.out = static_cast<uint16_t*>(y) + c0 * H;
    p.ldo = H;
    p.out_f32 = 0;
    if ((st = mlp_store(*dev, {cr, H, I, false, false, A, I, Wd, I, false},
                        p, LCE_K_MLP_DOWN, wsb + w.sync, s)) != LCE_OK)
      return st;
  }
  return LCE_OK;
}

lce_status lce_mlp_backward(const void* x, const void* Wg, const void* Wu,
                            const void* Wd, const void* dy, int64_t L,
                            int64_t H, int64_t I, int64_t chunk_rows,
                            void* dx, float* dWg, float* dWu, float* dWd,
                            void* ws, size_t ws_bytes, void* stream) {
  lce_status st = mlp_check(x, Wg, Wu, Wd, L, H, I);
  if (st != LCE_OK) return st;
  // dx, dWd and the pair (dWg, dWu) may each be NULL (not computed); dWg
  // and dWu come from one contraction, so both or neither; not all
  if (!dy || !ws || chunk_rows < 0 || (!dWg != !dWu) ||
      (!dx && !dWg && !dWd))
    return LCE_ERR_INVALID_ARG;
  const bool need_dgu = dx || dWg;  // dx and [dWg ; dWu] read [dg | du]
  if (!aligned16(dy) || !aligned16(dx) || !aligned16(dWg) ||
      !aligned16(dWu) || !aligned16(dWd) || !aligned16(ws))
    return LCE_ERR_INVALID_ARG;
  const MlpLayout w = mlp_layout(L, I, chunk_rows);
  if (ws_bytes < w.total) return LCE_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint16_t* G = reinterpret_cast<uint16_t*>(wsb + w.g);
  uint16_t* U = reinterpret_cast<uint16_t*>(wsb + w.u);
  uint16_t* A = reinterpret_cast<uint16_t*>(wsb + w.a);
  uint16_t* DGU = reinterpret_cast<uint16_t*>(wsb + w.dgu);
  for (int64_t c0 = 0; c0 < L; c0 += w.chunk) {
    const int64_t cr = std::min(w.chunk, L - c0);
    const uint16_t* xc = static_cast<const uint16_t*>(x) + c0 * H;
    const uint16_t* dyc = static_cast<const uint16_t*>(dy) + c0 * H;
    // (1) recompute g_c, u_c, a_c
    if ((st = mlp_gate_up(*dev, xc, cr, Wg, Wu, H, I, A, G, U, wsb + w.sync,
                          s)) != LCE_OK)
      return st;
    // (2) da_c = dy_c Wd -> dg_c, du_c into [dg | du]
    if (need_dgu) {
      GemmOperands o{cr, I, H, false, true, dyc, H, Wd, I, false};
      GemmPlan pl;
      if ((st = plan_gemm(o, *dev, &pl)) != LCE_OK) return st;
      SwigluBwdParams p{};
      if ((st = tmap_store_box(&p.map_dgu, DGU, 2 * I, cr, 2 * I)) != LCE_OK)
        return st;
      p.g = G;
      p.u = U;
      p.ld_gu = I;
      p.du_off = I;
      cudaError_t e = pace(&pl, wsb + w.sync, s);
      if (e != cudaSuccess) return cuda_fail(e, "pace");
      ProfScope ps(LCE_K_MLP_DA, s);
      e = launch_gemm_swiglu_bwd(pl.pair, pl.ta, pl.tb, pl.tb2, pl.g, p,
                                 dev->err, pl.grid, s);
      ps.done(2.0 * cr * I * H);
      if (e != cudaSuccess) return cuda_fail(e, "mlp_da");
    }
    // (3) dx_c = [dg | du] [Wg ; Wu]  (K = 2I, B from two maps along K)
    if (dx) {
      GemmOperands o{cr, H, 2 * I, false, true, DGU, 2 * I, Wg, H, false};
      o.b_dual = 2;
      o.b2 = Wu;
      o.k_split = I;
      StoreParams p{};
      p.out = static_cast<uint16_t*>(dx) + c0 * H;
      p.ldo = H;
      if ((st = mlp_store(*dev, o, p, LCE_K_MLP_DX, wsb + w.sync, s)) !=
          LCE_OK)
        return st;
    }
    // (4) dWd (+)= dy_c^T a_c
    if (dWd) {
      StoreParams p{};
      p.out = dWd;
      p.ldo = I;
      p.out_f32 = 1;
      p.accumulate = c0 > 0;
      if ((st = mlp_store(*dev, {H, I, cr, true, true, dyc, H, A, I, false},
                          p, LCE_K_MLP_DWD, wsb + w.sync, s)) != LCE_OK)
        return st;
    }
    // (5) [dWg ; dWu] (+)= [dg | du]^T x_c, rows >= I going to dWu
    if (dWg) {
      StoreParams p{};
      p.out = dWg;
      p.out2 = dWu;
      p.split_row = I;
      p.ldo = H;
      p.out_f32 = 1;
      p.accumulate = c0 > 0;
      if ((st = mlp_store(*dev, {2 * I, H, cr, true, true, DGU, 2 * I, xc, H,
                                 false},
                          p, LCE_K_MLP_DWGU, wsb + w.sync, s)) != LCE_OK)
        return st;
    }
  }
  return LCE_OK;
}

lce_status lce_get_error(void* stream) {
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  if ((e = cudaMemcpy(&word, dev->err, sizeof word, cudaMemcpyDeviceToHost)) !=
      cudaSuccess)
    return cuda_fail(e, "read error word");
  if (word) {
    const unsigned zero = 0;
    if ((e = cudaMemcpy(dev->err, &zero, sizeof zero,
                        cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear error word");
  }
  if (word & ERRBIT_TIMEOUT) return LCE_ERR_TIMEOUT;
  if (word & ERRBIT_LABEL_RANGE) return LCE_ERR_LABEL_RANGE;
  return LCE_OK;
}

const char* lce_status_string(lce_status s) {
  switch (s) {
    case LCE_OK: return "LCE_OK";
    case LCE_ERR_INVALID_ARG: return "LCE_ERR_INVALID_ARG";
    case LCE_ERR_UNSUPPORTED: return "LCE_ERR_UNSUPPORTED";
    case LCE_ERR_WORKSPACE: return "LCE_ERR_WORKSPACE";
    case LCE_ERR_LABEL_RANGE: return "LCE_ERR_LABEL_RANGE";
    case LCE_ERR_TIMEOUT: return "LCE_ERR_TIMEOUT";
    case LCE_ERR_CUDA: return "LCE_ERR_CUDA";
  }
  return "LCE_ERR_UNKNOWN";
}

const char* lce_last_cuda_error(void) { return t_last_cuda_error; }

lce_status lce_test_gemm(const void* A, const void* B, float* D, int64_t M,
                         int64_t N, int64_t K, int a_mn, int b_mn,
                         void* stream) {
  if (!A || !B || !D) return LCE_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || K < 1 || N % 8 || M > (1ll << 30) ||
      N > (1ll << 30) || K > (1ll << 30))
    return LCE_ERR_INVALID_ARG;
  if ((a_mn ? M : K) % 8 || (b_mn ? N : K) % 8) return LCE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D))
    return LCE_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  GemmPlan pl;
  if ((st = plan_gemm({M, N, K, a_mn != 0, b_mn != 0, A, a_mn ? M : K, B,
                       b_mn ? N : K, false},
                      *dev, &pl)) != LCE_OK)
    return st;
  StoreParams p{};
  p.out = D;
  p.ldo = N;
  p.out_f32 = 1;
  p.accumulate = 0;
  p.dloss = nullptr;
  p.n_valid = nullptr;
  ProfScope ps(LCE_K_TEST_GEMM, static_cast<cudaStream_t>(stream));
  cudaError_t e = run_store(pl, a_mn != 0, b_mn != 0, p, dev->err,
                            static_cast<cudaStream_t>(stream));
  ps.done(2.0 * M * N * K);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "test_gemm");
}

lce_status lce_test_wait_timeout(uint64_t timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return LCE_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  ProfScope ps(LCE_K_WAIT_PROBE, static_cast<cudaStream_t>(stream));
  cudaError_t e = launch_wait_probe(dev->err, timeout_ns,
                                    static_cast<cudaStream_t>(stream));
  ps.done(0);
  return e == cudaSuccess ? LCE_OK : cuda_fail(e, "wait_probe");
}

lce_status lce_set_cta_pair(int enable) {
  if (enable != 0 && enable != 1) return LCE_ERR_INVALID_ARG;
  g_pair_mode.store(enable);
  return LCE_OK;
}

int lce_get_cta_pair(void) { return use_pair() ? 1 : 0; }

lce_status lce_set_wave_sync(int enable) {
  if (enable != 0 && enable != 1) return LCE_ERR_INVALID_ARG;
  g_wave_mode.store(enable);
  return LCE_OK;
}

int lce_get_wave_sync(void) { return wave_sync_on() ? 1 : 0; }

lce_status lce_profile_start(void) {
  if (t_prof.on) return LCE_ERR_INVALID_ARG;
  t_prof.recs.clear();
  t_prof.used = 0;
  t_prof.on = true;
  return LCE_OK;
}

lce_status lce_profile_stop(lce_kernel_stat* stats) {
  if (!t_prof.on || !stats) return LCE_ERR_INVALID_ARG;
  t_prof.on = false;
  for (int k = 0; k < LCE_KERNEL_KINDS; ++k) {
    stats[k].name = kKindNames[k];
    stats[k].launches = 0;
    stats[k].total_ms = 0.0;
    stats[k].flops = 0.0;
  }
  lce_status st = LCE_OK;
  for (const ProfRec& r : t_prof.recs) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.e0, r.e1);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "profile events");
      continue;
    }
    stats[r.kind].launches += 1;
    stats[r.kind].total_ms += ms;
    stats[r.kind].flops += r.flops;
  }
  t_prof.recs.clear();
  t_prof.used = 0;
  return st;
}

lce_status lce_forward_static(const void* h, const void* W,
                              const int64_t* labels, int64_t L, int64_t H,
                              int64_t V, int64_t ignore_index, float* loss,
                              float* lse, void* stream) {
  if (!h || !W || !labels || !loss || !lse) return LCE_ERR_INVALID_ARG;
  if (!sizes_ok(L, H, V)) return LCE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(W) ||
      (reinterpret_cast<uintptr_t>(labels) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(loss) & 3u))
    return LCE_ERR_INVALID_ARG;
  if (L > kStaticMaxRows) {
    std::snprintf(t_last_cuda_error, sizeof t_last_cuda_error,
                  "lce_forward_static: L = %lld exceeds the static scratch "
                  "limit of %lld rows",
                  static_cast<long long>(L),
                  static_cast<long long>(kStaticMaxRows));
    return LCE_ERR_WORKSPACE;
  }
  DeviceInfo* dev = nullptr;
  lce_status st = device_info(&dev);
  if (st != LCE_OK) return st;
  void* scratch = nullptr;
  if ((st = static_scratch(&scratch)) != LCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // carve the scratch
  uint8_t* base = static_cast<uint8_t*>(scratch);
  const int64_t nb = ceil_div(L, 256);
  const size_t off_sums = 256;
  const size_t off_zy = static_cast<size_t>(round_up(off_sums + nb * 8, 256));
  const size_t off_part = static_cast<size_t>(round_up(off_zy + L * 4, 256));
  const size_t part_bytes = static_cast<size_t>(round_up(L * 4, 256));
  const int max_splits = static_cast<int>(
      std::min<size_t>(kMaxSplits,
                       (kStaticScratchBytes - off_part) / (2 * part_bytes)));
  auto* n_valid = reinterpret_cast<unsigned long long*>(base);
  double* block_sums = reinterpret_cast<double*>(base + off_sums);

  // the valid-row count starts at zero on every call (a memset, not an
  // allocation); every other region is written before it is read
  cudaError_t e =
      launch_count_valid(labels, L, V, ignore_index, n_valid, dev->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "count_valid");

  const int num_m = static_cast<int>(ceil_div(L, BM));
  const int num_n = static_cast<int>(ceil_div(V, BN));
  int splits = 1, tps = num_n;
  choose_splits(num_m, num_n, dev->num_sms, H, &splits, &tps);
  if (splits > max_splits) {
    tps = static_cast<int>(ceil_div(num_n, max_splits));
    splits = static_cast<int>(ceil_div(num_n, tps));
  }
  const GemmGeom g = make_geom(L, V, H, splits, tps);
  CUtensorMap ta, tb;
  if ((st = tmap_kmajor(&ta, h, H, L, H, BM)) != LCE_OK) return st;
  if ((st = tmap_kmajor(&tb, W, H, V, H, BN)) != LCE_OK) return st;
  LseParams p{};
  p.labels = labels;
  p.zy = reinterpret_cast<float*>(base + off_zy);
  p.part_m = reinterpret_cast<float*>(base + off_part);
  p.part_s = reinterpret_cast<float*>(base + off_part + splits * part_bytes);
  p.ignore_index = ignore_index;
  if ((e = launch_gemm_lse(ta, tb, g, p, dev->err, grid_for(g, dev->num_sms),
                           s)) != cudaSuccess)
    return cuda_fail(e, "gemm_lse");
  int nblocks = 0;
  if ((e = launch_lse_combine(p.part_m, p.part_s, g.splits, p.zy, labels, L, V,
                              ignore_index, lse, block_sums, &nblocks, s)) !=
      cudaSuccess)
    return cuda_fail(e, "lse_combine");
  if ((e = launch_loss_finalize(block_sums, nblocks, n_valid, loss, s)) !=
      cudaSuccess)
    return cuda_fail(e, "loss_finalize");
  return LCE_OK;
}

}  // extern "C"
