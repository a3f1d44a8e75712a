// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument checks, TMA
// tensor-map encoding, the persistent launch and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fa.h"
#include "fa_fwd_1tile_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_fwd_row_kernel.cuh"
#include "fa_merge_kernel.cuh"

// Built-in scratch for fa_fwd_splitkv_noalloc: callers that may not allocate device
// memory get the split-KV workspace from this fixed array instead.  It is part of the
// library's device image, so every GPU that loads the library holds it until exit.
constexpr size_t kStaticScratchBytes = size_t{64} << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kVersion = 300;  // 0.3.0 (fa_fwd_options gained `block_kv`)
constexpr int kMaxDevices = 64;
constexpr long long kDefaultBudget = 2000000000LL;  // ~1 s of SM clock

thread_local std::string t_last_error;

int set_error(int status, const std::string& msg) {
  t_last_error = msg;
  return status;
}

int cuda_error(const char* what, cudaError_t e) {
  return set_error(FA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled, fetched through the runtime so the library needs no -lcuda
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool probed = false;
  bool arch_ok = false;
  int num_sms = 0;
  bool smem_set[5][2] = {};                                    // two-tile kernel, per head dim and key tile
  bool smem_set_one[5] = {false, false, false, false, false};  // one-tile kernel
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int head_dim_index(int64_t d) {
  switch (d) {
    case 16: return 0;
    case 32: return 1;
    case 64: return 2;
    case 128: return 3;
    case 256: return 4;
    default: return -1;
  }
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Encode a [BH, N, d] bf16 tensor as a 3-D tiled map with a (W x rows x 1) box: 128 rows
// for Q tiles, the key-tile width for K and V.
int encode_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t d,
               int rows = fa_sm103::kBlockM) {
  const int w = d < 64 ? static_cast<int>(d) : 64;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2),
                                 static_cast<cuuint64_t>(N * d * 2)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(w), static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = w * 2 == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : w * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return set_error(FA_ERR_CUDA, buf);
  }
  return FA_OK;
}

constexpr int kMaxSplits = 64;

int64_t units_for(int64_t BH, int64_t N) {
  return ((N + fa_sm103::kUnitRows - 1) / fa_sm103::kUnitRows) * BH;
}

// Bytes of workspace a split launch needs: per item 256 rows of normalised partial O
// (fp32, d per row) and 256 partial logsumexps.
int64_t workspace_bytes(int64_t BH, int64_t N, int64_t d, int splits) {
  if (splits <= 1) return 0;
  const int64_t rows = units_for(BH, N) * splits * fa_sm103::kUnitRows;
  return rows * d * 4 + rows * 4;
}

// Split only when the longest unit would be the critical path -- its key tiles exceed
// twice the average work per SM -- and that average is large enough (>= 16 tiles) to
// amortise a piece's fixed costs and the merge.  Pieces are ~1.5x the average.
// (Measured on GB300, B1 d128 causal: H1 N32768 548 -> 946 TFLOP/s and H4 N8192
// 515 -> 644 TFLOP/s with two pieces; H8 N4096 and B1 H32 N2048 are faster unsplit.)
int choose_splits(int64_t BH, int64_t N, int num_sms, int causal) {
  const int64_t nqb = (N + fa_sm103::kUnitRows - 1) / fa_sm103::kUnitRows;
  const int64_t nkv = (N + fa_sm103::kBlockN - 1) / fa_sm103::kBlockN;
  const int64_t n_max = causal ? (2 * nqb < nkv ? 2 * nqb : nkv) : nkv;
  // key tiles over all units (a unit does max(n0, n1) tile steps)
  int64_t total = 0;
  for (int64_t qb = 0; qb < nqb; ++qb) total += causal ? (2 * qb + 2 < nkv ? 2 * qb + 2 : nkv) : nkv;
  total *= BH;
  const double per_sm = static_cast<double>(total) / num_sms;
  if (n_max <= 2.0 * per_sm || per_sm < 16.0) return 1;
  int64_t sp = static_cast<int64_t>(std::ceil(static_cast<double>(n_max) / (1.5 * per_sm)));
  if (sp > kMaxSplits) sp = kMaxSplits;
  return sp < 1 ? 1 : static_cast<int>(sp);
}

// Workspace large enough for `splits` and clear of every tensor (sets the error text).
bool workspace_fits(const void* ws, size_t size, int64_t BH, int64_t N, int64_t d, int splits,
                    const void* q, const void* k, const void* v, const void* o, size_t bytes,
                    const void* lse, size_t lse_bytes) {
  const int64_t need = workspace_bytes(BH, N, d, splits);
  if (static_cast<int64_t>(size) < need) {
    set_error(FA_ERR_INVALID_ARG, "workspace too small (see fa_splitkv_workspace_bytes)");
    return false;
  }
  for (const void* t : {q, k, v, o})
    if (overlaps(ws, static_cast<size_t>(need), t, bytes)) {
      set_error(FA_ERR_INVALID_ARG, "workspace overlaps a tensor");
      return false;
    }
  if (lse && overlaps(ws, static_cast<size_t>(need), lse, lse_bytes)) {
    set_error(FA_ERR_INVALID_ARG, "workspace overlaps lse");
    return false;
  }
  return true;
}

// Heads per scheduling group: their K and V together take at most ~64 MB of L2.
int64_t group_heads_for(int64_t BH, int64_t N, int64_t d) {
  const int64_t kv_bytes_per_head = 2 * N * d * 2;
  int64_t g = (int64_t{64} << 20) / (kv_bytes_per_head > 0 ? kv_bytes_per_head : 1);
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return g;
}

// ---- kernel choice ------------------------------------------------------------------
// At head dims 32 to 128 both kernels serve a call.  The two-tile kernel's 256-row units
// share each K/V tile between two Q tiles and run a step 1.14-1.18x faster; the one-tile
// kernel's 128-row units are half as long, which matters when there are few units per
// SM: under the causal mask unit lengths run from 1 to N/128 key tiles, and the longest
// units set the finishing time.  The choice replays the static schedule both kernels
// follow (unit_coords / item_of: grouped longest-first order handed out in snakes, each
// kernel at its better item order) and compares the busiest CTA's total.  Cost unit:
// one (128-row Q tile x 128-key tile) step of the two-tile kernel.
struct CostModel {
  double two_unit;      // fixed cost of an unsplit two-tile unit
  double one_unit;      // fixed cost of a one-tile unit, in one-tile steps
  double one_step;      // a one-tile kernel step, in two-tile steps
  double split_piece;   // fixed cost of one split piece
  double merge_fixed;   // the merge launch
  double merge_per_mb;  // per MB of fp32 partial outputs (written, merged)
  double one_piece;     // fixed cost of a one-tile split piece, in one-tile steps
};
// Fitted to GB300 timings of the current kernels, per head dim: both kernels unsplit on
// 46 shapes (B*H 1-64, N 256-65536, causal and not) and split 2, 3, 4, 5, 6 and 8 ways on
// the 21 of them with at most 152 two-tile or 304 one-tile units (d = 256: the one-tile
// kernel on 16 shapes).  The constants were chosen on a grid to minimise the time lost to
// wrong picks, replaying this planner exactly: its pick is within 2 % of the fastest
// measured launch on 45 of 46 shapes at d = 128 (the other 2.2 %), all 46 at d = 64, 45
// of 46 at d = 32 (the other 5.9 %) and 15 of 16 at d = 256 (2.6 %).  The split costs at
// d = 128 were refitted once more after the merge kernel got faster (a half-warp per row
// for up to four pieces); d = 32, 64 and 256 keep the fit to the earlier merge.  At d =
// 256 only the one-tile kernel runs: its step is the unit.
constexpr CostModel kCostD128 = {3.0, 1.0, 1.07, 12.0, 0.0, 0.25, 6.0};
constexpr CostModel kCostD64 = {8.0, 2.0, 1.30, 8.0, 15.0, 0.25, 1.0};
constexpr CostModel kCostD32 = {8.0, 2.0, 1.30, 4.0, 20.0, 0.25, 1.0};
constexpr CostModel kCostD256 = {0.0, 0.0, 1.0, 0.0, 0.0, 0.25, 3.0};
constexpr int kModelMaxSms = 1024;
constexpr int64_t kModelUnitsPerSm = 4;      // more 256-row units per SM: two-tile kernel
constexpr int64_t kModelMaxItems = 1 << 16;  // bound on the replayed schedule's length

// The cost table of a head dim the planner models (32-256), else null (16: two-tile only).
const CostModel* cost_model(int64_t d) {
  if (d == 256) return &kCostD256;
  if (d == 128) return &kCostD128;
  if (d == 64) return &kCostD64;
  if (d == 32) return &kCostD32;
  return nullptr;
}

struct Plan {
  int kernel;  // FA_KERNEL_TWO_TILE or FA_KERNEL_ONE_TILE
  int splits;
};

// Key tiles a Q tile starting at row_start visits (the kernels' tiles_for).
int64_t tiles_from(int64_t row_start, int64_t N, int64_t nkv, int causal) {
  if (row_start >= N) return 0;
  if (!causal) return nkv;
  const int64_t t = row_start / fa_sm103::kBlockN + 1;
  return t < nkv ? t : nkv;
}

// Query block (in units of `unit_rows`) of unit u in the grouped longest-first order.
int64_t unit_block(int64_t u, int64_t BH, int64_t nqb, int64_t gh) {
  const int64_t g = u / (gh * nqb);
  const int64_t heads = std::min(gh, BH - g * gh);
  return nqb - 1 - (u - g * gh * nqb) / heads;
}

// Order 2's per-group CTA offset: the CTAs a full group's part-filled last round used
// (positions 0..rem-1 on an even round, G-rem..G-1 on an odd one) are skipped.
int group_shift(int64_t group_items, int grid) {
  const int64_t last = group_items / grid, rem = group_items % grid;
  if (rem == 0) return 0;
  return static_cast<int>((last & 1) ? grid - rem : rem);
}

// The busiest CTA's total cost when `items` items (costs cost(i), numbered as item_of
// numbers them) are handed out over `grid` CTAs in item order `order` (item_of inverted:
// item i of a group sits at round i / grid, position i % grid; order 0 is one group).
template <class Cost>
double schedule_makespan(int64_t items, int grid, int order, int64_t group_items, Cost cost) {
  double load[kModelMaxSms] = {};
  const int64_t span = order == 0 ? items : group_items;
  const int shift = group_shift(group_items, grid);
  int64_t g = 0;
  for (int64_t base = 0; base < items; base += span, ++g) {
    const int64_t n = std::min(span, items - base);
    const int off = static_cast<int>(g * shift % grid);
    for (int64_t i = 0; i < n; ++i) {
      const int64_t k = i / grid;
      const int r = static_cast<int>(i - k * grid);
      const int c = (k & 1) ? grid - 1 - r : r;
      const int cta = order == 1 ? ((g & 1) ? grid - 1 - c : c) : order == 2 ? (c + off) % grid : c;
      load[cta] += cost(base + i);
    }
  }
  return *std::max_element(load, load + grid);
}

double model_two_tile(const CostModel& cm, int64_t BH, int64_t N, int64_t d, int causal, int grid,
                      int splits, int order) {
  const int64_t nqb = (N + fa_sm103::kUnitRows - 1) / fa_sm103::kUnitRows;
  const int64_t nkv = (N + fa_sm103::kBlockN - 1) / fa_sm103::kBlockN;
  const int64_t gh = group_heads_for(BH, N, d);
  const int64_t items = nqb * BH * splits;
  double t = schedule_makespan(items, grid, order, gh * nqb * splits, [&](int64_t w) {
    const int64_t u = w / splits, sp = w - u * splits;
    const int64_t row0 = unit_block(u, BH, nqb, gh) * fa_sm103::kUnitRows;
    const int64_t n0 = tiles_from(row0, N, nkv, causal);
    const int64_t n1 = tiles_from(row0 + fa_sm103::kBlockM, N, nkv, causal);
    const int64_t n = std::max(n0, n1);
    const int64_t k0 = sp * n / splits, k1 = (sp + 1) * n / splits;
    if (k1 <= k0) return 0.0;
    const double steps = static_cast<double>(std::max<int64_t>(0, std::min(n0, k1) - k0) +
                                             std::max<int64_t>(0, std::min(n1, k1) - k0));
    return steps + (splits > 1 ? cm.split_piece : cm.two_unit);
  });
  if (splits > 1)
    t += cm.merge_fixed + cm.merge_per_mb * static_cast<double>(splits * BH * N * d * 4) * 1e-6;
  return t;
}

double model_one_tile(const CostModel& cm, int64_t BH, int64_t N, int64_t d, int causal, int grid,
                      int order, int splits = 1) {
  const int64_t nqb = (N + fa_sm103::one::kUnitRows1 - 1) / fa_sm103::one::kUnitRows1;
  const int64_t nkv = (N + fa_sm103::kBlockN - 1) / fa_sm103::kBlockN;
  const int64_t gh = group_heads_for(BH, N, d);
  const int64_t items = nqb * BH * splits;
  double t = cm.one_step * schedule_makespan(items, grid, order, gh * nqb * splits, [&](int64_t w) {
    const int64_t u = w / splits, sp = w - u * splits;
    const int64_t row0 = unit_block(u, BH, nqb, gh) * fa_sm103::one::kUnitRows1;
    const int64_t n = tiles_from(row0, N, nkv, causal);
    const int64_t k0 = sp * n / splits, k1 = (sp + 1) * n / splits;
    if (k1 <= k0) return 0.0;
    return static_cast<double>(k1 - k0) + (splits > 1 ? cm.one_piece : cm.one_unit);
  });
  if (splits > 1)
    t += cm.merge_fixed + cm.merge_per_mb * static_cast<double>(splits * BH * N * d * 4) * 1e-6;
  return t;
}

// The item order (Params::order) with the shortest modelled makespan for a launch of
// `kernel` on `grid` CTAs.  The orders differ only with two or more head groups.  One
// snake over everything starts each group mid-round; a snake per group fixes that (b1
// h32 S8192, two groups of 3.4 rounds: 1154 -> 1266 TFLOP/s on GB300), mirrored in odd
// groups (best with two groups) or shifted past each predecessor's part-filled last
// round (best with many: b8 h32 S16384 +1.4 %, d256 b4 h16 S8192 1554 TFLOP/s with each
// group's K and V together in L2).  Decisions are kept in a small cache, so repeated
// shapes replay the schedules once.
constexpr int64_t kOrderMaxItems = int64_t{1} << 20;
struct OrderEntry {
  int64_t BH, N, d;
  int causal, grid, splits, kernel, order;
  bool valid;
};
std::mutex g_order_mu;
OrderEntry g_order_cache[32];
int g_order_next = 0;

int schedule_order(int kernel, int64_t BH, int64_t N, int64_t d, int causal, int grid, int splits) {
  const int64_t gh = group_heads_for(BH, N, d);
  const int64_t rows = kernel == FA_KERNEL_ONE_TILE ? fa_sm103::one::kUnitRows1 : fa_sm103::kUnitRows;
  const int64_t items = (N + rows - 1) / rows * BH * splits;
  if (gh >= BH || grid > kModelMaxSms || items > kOrderMaxItems) return 0;
  causal = causal ? 1 : 0;
  {
    std::lock_guard<std::mutex> lock(g_order_mu);
    for (const OrderEntry& e : g_order_cache)
      if (e.valid && e.BH == BH && e.N == N && e.d == d && e.causal == causal && e.grid == grid &&
          e.splits == splits && e.kernel == kernel)
        return e.order;
  }
  const CostModel& cm = cost_model(d) ? *cost_model(d) : kCostD128;
  double t[3];
  for (int o = 0; o < 3; ++o)
    t[o] = kernel == FA_KERNEL_ONE_TILE ? model_one_tile(cm, BH, N, d, causal, grid, o, splits)
                                         : model_two_tile(cm, BH, N, d, causal, grid, splits, o);
  int order = 0;
  for (int o = 1; o < 3; ++o)
    if (t[o] < t[order]) order = o;
  std::lock_guard<std::mutex> lock(g_order_mu);
  g_order_cache[g_order_next] = {BH, N, d, causal, grid, splits, kernel, order, true};
  g_order_next = (g_order_next + 1) % 32;
  return order;
}

// Split counts the planner also models when there are few units per SM (one or two
// heads at N <= 16384 run fastest split 3 to 6 ways, which the heuristic of choose_splits
// never proposes there).
constexpr int kSplitCandidates[] = {2, 3, 4, 5, 6, 8};

// The launch for a non-empty problem.  max_splits: the most key-range pieces the call
// can hold partial results for (1 = no workspace).  Candidates: the two-tile kernel
// unsplit, split as choose_splits says and (with no more 256-row units than SMs) split
// 2-8 ways; the one-tile kernel unsplit and (with at most two 128-row units per SM)
// split 2-8 ways.  Each is modelled at its better item order; the shortest wins.
Plan plan_for(int64_t BH, int64_t N, int64_t d, int causal, int sms, int max_splits) {
  const bool two_ok = d <= 128, one_ok = d >= 32;
  int heur = (max_splits > 1 && two_ok) ? choose_splits(BH, N, sms, causal) : 1;
  if (heur > max_splits) heur = max_splits;
  const int64_t units = units_for(BH, N);
  const int64_t units1 = (N + fa_sm103::one::kUnitRows1 - 1) / fa_sm103::one::kUnitRows1 * BH;
  const CostModel* cm = cost_model(d);
  if (!cm || sms > kModelMaxSms || units > kModelUnitsPerSm * sms ||
      units1 * std::max(heur, 8) > kModelMaxItems)
    return two_ok ? Plan{FA_KERNEL_TWO_TILE, heur} : Plan{FA_KERNEL_ONE_TILE, 1};
  Plan best = {0, 0};
  double t_best = 0.0;
  auto consider = [&](int kernel, int splits) {
    if (splits < 1 || splits > max_splits) return;
    const int64_t items = (kernel == FA_KERNEL_ONE_TILE ? units1 : units) * splits;
    const int grid = static_cast<int>(std::min<int64_t>(sms, items));
    double t = 0.0;
    for (int o = 0; o < 3; ++o) {
      const double to = kernel == FA_KERNEL_ONE_TILE
                            ? model_one_tile(*cm, BH, N, d, causal, grid, o, splits)
                            : model_two_tile(*cm, BH, N, d, causal, grid, splits, o);
      t = o == 0 ? to : std::min(t, to);
    }
    if (best.kernel == 0 || t < t_best) {
      t_best = t;
      best = {kernel, splits};
    }
  };
  if (two_ok) {
    consider(FA_KERNEL_TWO_TILE, 1);
    if (heur > 1) consider(FA_KERNEL_TWO_TILE, heur);
    if (units <= sms)
      for (const int sp : kSplitCandidates) consider(FA_KERNEL_TWO_TILE, sp);
  }
  if (one_ok) {
    consider(FA_KERNEL_ONE_TILE, 1);
    if (units1 <= 2 * sms)
      for (const int sp : kSplitCandidates) consider(FA_KERNEL_ONE_TILE, sp);
  }
  return best;
}

// plan_for's decisions, kept per shape: replaying the schedules of all candidates costs
// up to a millisecond of host time, which a loop of short launches must not pay per call.
struct PlanEntry {
  int64_t BH, N, d;
  int causal, sms, max_splits;
  Plan plan;
  bool valid;
};
std::mutex g_plan_mu;
PlanEntry g_plan_cache[64];
int g_plan_next = 0;

Plan plan_cached(int64_t BH, int64_t N, int64_t d, int causal, int sms, int max_splits) {
  causal = causal ? 1 : 0;
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (const PlanEntry& e : g_plan_cache)
      if (e.valid && e.BH == BH && e.N == N && e.d == d && e.causal == causal && e.sms == sms &&
          e.max_splits == max_splits)
        return e.plan;
  }
  const Plan pl = plan_for(BH, N, d, causal, sms, max_splits);
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plan_cache[g_plan_next] = {BH, N, d, causal, sms, max_splits, pl, true};
  g_plan_next = (g_plan_next + 1) % 64;
  return pl;
}

// The most pieces whose partial results fit `bytes` of workspace (1 if none fit).
int splits_fitting(int64_t BH, int64_t N, int64_t d, int64_t bytes) {
  int s = kMaxSplits;
  while (s > 1 && workspace_bytes(BH, N, d, s) > bytes) --s;
  return s;
}

// Fields every launch shares.  `unit_rows` = query rows per work unit (256 for the
// two-tile kernel, 128 for the head-dim-256 kernel).
fa_sm103::Params base_params(void* o, float* lse, int64_t BH, int64_t N, int64_t d, int unit_rows,
                             int causal, float scale, const fa_fwd_options* opts) {
  fa_sm103::Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = static_cast<int>(BH);
  p.N = static_cast<int>(N);
  p.nkv = static_cast<int>((N + fa_sm103::kBlockN - 1) / fa_sm103::kBlockN);
  p.nqb = static_cast<int>((N + unit_rows - 1) / unit_rows);
  p.num_units = static_cast<int>(static_cast<int64_t>(p.nqb) * BH);
  p.splits = 1;
  p.num_items = p.num_units;
  p.ws_o = nullptr;
  p.ws_lse = nullptr;
  p.group_heads = static_cast<int>(group_heads_for(BH, N, d));
  p.causal = causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.budget = (opts && opts->wait_budget_cycles > 0) ? opts->wait_budget_cycles : kDefaultBudget;
  p.inject = opts ? opts->inject_skip_kv_load : 0;
  return p;
}

// The item order (Params::order) and the rounds every role iterates over, for `grid` CTAs.
void set_schedule(fa_sm103::Params& p, int grid, int order) {
  p.order = order;
  p.group_items = p.group_heads * p.nqb * p.splits;
  p.group_shift = group_shift(p.group_items, grid);
  if (order == 0) {
    p.rounds_per_group = 0;
    p.num_rounds = (p.num_items + grid - 1) / grid;
  } else {
    const int groups = (p.BH + p.group_heads - 1) / p.group_heads;
    p.rounds_per_group = (p.group_items + grid - 1) / grid;
    p.num_rounds = groups * p.rounds_per_group;
  }
}

// The item order of a launch: pinned by opts->order, else schedule_order's choice.
int pick_order(const fa_fwd_options* opts, int kernel, int64_t BH, int64_t N, int64_t d, int causal,
               int grid, int splits) {
  if (opts && opts->order == FA_ORDER_ONE_SNAKE) return 0;
  if (opts && opts->order == FA_ORDER_GROUP_SNAKES) return 1;
  if (opts && opts->order == FA_ORDER_SHIFTED_SNAKES) return 2;
  return schedule_order(kernel, BH, N, d, causal, grid, splits);
}

int grid_for(const DeviceState& dev, const fa_fwd_options* opts, int items) {
  int grid = dev.num_sms;
  if (opts && opts->max_ctas > 0 && opts->max_ctas < grid) grid = opts->max_ctas;
  return grid > items ? items : grid;
}

// The merge of a split launch: one warp per query row; the partial outputs of up to
// 2 or 8 pieces are loaded up front (the smallest bucket that holds `splits`).
template <int HD, int UNIT_ROWS, int BN = fa_sm103::kBlockN>
int launch_merge(const fa_sm103::Params& p, int64_t BH, int64_t N, cudaStream_t stream) {
  constexpr int T = fa_sm103::kMergeThreads, WPB = T / 32;
  const int64_t rows = BH * N;
  auto blocks = [&](int rows_per_warp) {
    return static_cast<unsigned>((rows + int64_t{WPB} * rows_per_warp - 1) / (int64_t{WPB} * rows_per_warp));
  };
  // up to four pieces at head dims up to 128: a half-warp per row (65,536 rows x 2 pieces:
  // 19.5 -> 13.8 us; x 4: 16.4 -> 13.4 us); with 5-8 pieces the partials held per lane make
  // it slower than a warp per row
  if constexpr (HD <= 128) {
    if (p.splits <= 4) {
      if (p.splits <= 2)
        fa_sm103::fa_merge2_kernel<HD, UNIT_ROWS, BN, 2><<<blocks(2), T, 0, stream>>>(p);
      else
        fa_sm103::fa_merge2_kernel<HD, UNIT_ROWS, BN, 4><<<blocks(2), T, 0, stream>>>(p);
      const cudaError_t e = cudaGetLastError();
      return e != cudaSuccess ? cuda_error("merge kernel launch", e) : FA_OK;
    }
  }
  if (p.splits <= 2)
    fa_sm103::fa_merge_kernel<HD, UNIT_ROWS, 2, BN, 1><<<blocks(1), T, 0, stream>>>(p);
  else if (p.splits <= 8)
    fa_sm103::fa_merge_kernel<HD, UNIT_ROWS, 8, BN, 1><<<blocks(1), T, 0, stream>>>(p);
  else
    fa_sm103::fa_merge_kernel<HD, UNIT_ROWS, 0, BN, 1><<<blocks(1), T, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error("merge kernel launch", e);
  return FA_OK;
}

// ---- register split of the two-tile kernel ------------------------------------------
// fa_fwd_row_kernel moves registers between its warpgroups with setmaxnreg (softmax up,
// epilogue and control down); the shares add up to exactly the registers the block is
// launched with, 512 threads x kLaunchRegs.  setmaxnreg.inc waits until the block's pool
// can satisfy it, and that wait has no bound: a build whose per-thread allocation differs
// (another compiler release, -G, -maxrregcount) would leave the softmax warpgroups waiting
// forever, outside every bounded barrier wait of the kernel.  So the compiled allocation
// is checked before the first launch, and a mismatch refuses the launch.
std::atomic<int> g_regs_override{0};  // test hook: > 0 stands in for the compiled count

int register_split_check(int num_regs, int max_threads) {
  using namespace fa_sm103::rowk;
  if (num_regs == kLaunchRegs && max_threads >= kThreadsR) return FA_OK;
  char buf[240];
  snprintf(buf, sizeof buf,
           "fa_fwd_row_kernel was compiled to %d registers per thread (at most %d threads per "
           "block); its setmaxnreg split needs exactly %d with %d threads, so it is not launched",
           num_regs, max_threads, kLaunchRegs, kThreadsR);
  return set_error(FA_ERR_UNSUPPORTED, buf);
}

template <int HD, int BN>
int check_row_kernel_registers() {
  const void* fns[2] = {reinterpret_cast<const void*>(fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, false>),
                        reinterpret_cast<const void*>(fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, true>)};
  for (const void* fn : fns) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, fn);
    if (e != cudaSuccess) return cuda_error("cudaFuncGetAttributes", e);
    const int fake = g_regs_override.load();
    const int st = register_split_check(fake > 0 ? fake : a.numRegs, a.maxThreadsPerBlock);
    if (st != FA_OK) return st;
  }
  return FA_OK;
}

// The two-tile kernel (256-row units) with key tiles of BN keys (128, or 64 on request).
template <int HD, int BN>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH,
           int64_t N, int causal, float scale, cudaStream_t stream, const DeviceState& dev,
           bool& smem_set, const fa_fwd_options* opts, int splits, void* workspace) {
  CUtensorMap mq, mk, mv;
  int st;
  // the first launch per device, head dim and key tile (and every launch while the test
  // hook is set)
  if ((!smem_set || g_regs_override.load() > 0) && (st = check_row_kernel_registers<HD, BN>()) != FA_OK)
    return st;
  if ((st = encode_map(&mq, q, BH, N, HD)) != FA_OK) return st;
  if ((st = encode_map(&mk, k, BH, N, HD, BN)) != FA_OK) return st;
  if ((st = encode_map(&mv, v, BH, N, HD, BN)) != FA_OK) return st;
  if (!smem_set) {
    cudaError_t e = cudaFuncSetAttribute(fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fa_sm103::rowk::row_kernel_smem<HD, BN, false>());
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               fa_sm103::rowk::row_kernel_smem<HD, BN, true>());
    if (e != cudaSuccess) return cuda_error("cudaFuncSetAttribute", e);
    smem_set = true;
  }
  fa_sm103::Params p = base_params(o, lse, BH, N, HD, fa_sm103::kUnitRows, causal, scale, opts);
  p.nkv = static_cast<int>((N + BN - 1) / BN);
  p.splits = splits;
  p.num_items = p.num_units * splits;
  p.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_lse = splits > 1 ? static_cast<float*>(workspace) +
                              static_cast<size_t>(p.num_items) * fa_sm103::kUnitRows * HD
                        : nullptr;
  const int grid = grid_for(dev, opts, p.num_items);
  set_schedule(p, grid, pick_order(opts, FA_KERNEL_TWO_TILE, BH, N, HD, causal, grid, splits));
  constexpr int kThr = fa_sm103::rowk::kThreadsR;
  if (splits > 1)
    fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, true>
        <<<grid, kThr, fa_sm103::rowk::row_kernel_smem<HD, BN, true>(), stream>>>(mq, mk, mv, p);
  else
    fa_sm103::rowk::fa_fwd_row_kernel<HD, BN, false>
        <<<grid, kThr, fa_sm103::rowk::row_kernel_smem<HD, BN, false>(), stream>>>(mq, mk, mv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error("kernel launch", e);
  if (splits > 1) return launch_merge<HD, fa_sm103::kUnitRows, BN>(p, BH, N, stream);
  return FA_OK;
}

// The one-Q-tile kernel (128-row units): head dims 32 to 256, split or not.  A split
// launch writes per-piece partial results to the workspace (items x 128 rows: partial O
// then partial lse) and the merge kernel combines them.
template <int HD>
int launch_one(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH,
               int64_t N, int causal, float scale, cudaStream_t stream, const DeviceState& dev,
               bool& smem_set, const fa_fwd_options* opts, int splits, void* workspace) {
  constexpr int SMEM = fa_sm103::one::Cfg1<HD>::SMEM_BYTES;
  CUtensorMap mq, mk, mv;
  int st;
  if ((st = encode_map(&mq, q, BH, N, HD)) != FA_OK) return st;
  if ((st = encode_map(&mk, k, BH, N, HD)) != FA_OK) return st;
  if ((st = encode_map(&mv, v, BH, N, HD)) != FA_OK) return st;
  if (!smem_set) {
    cudaError_t e = cudaFuncSetAttribute(fa_sm103::one::fa_fwd_1tile_kernel<HD, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_sm103::one::fa_fwd_1tile_kernel<HD, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return cuda_error("cudaFuncSetAttribute", e);
    smem_set = true;
  }
  fa_sm103::Params p =
      base_params(o, lse, BH, N, HD, fa_sm103::one::kUnitRows1, causal, scale, opts);
  p.splits = splits;
  p.num_items = p.num_units * splits;
  p.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_lse = splits > 1 ? static_cast<float*>(workspace) +
                              static_cast<size_t>(p.num_items) * fa_sm103::one::kUnitRows1 * HD
                        : nullptr;
  const int grid = grid_for(dev, opts, p.num_items);
  set_schedule(p, grid, pick_order(opts, FA_KERNEL_ONE_TILE, BH, N, HD, causal, grid, splits));
  constexpr int kThr = fa_sm103::one::kThreads1;
  if (splits > 1)
    fa_sm103::one::fa_fwd_1tile_kernel<HD, true><<<grid, kThr, SMEM, stream>>>(mq, mk, mv, p);
  else
    fa_sm103::one::fa_fwd_1tile_kernel<HD, false><<<grid, kThr, SMEM, stream>>>(mq, mk, mv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error("kernel launch", e);
  if (splits > 1) return launch_merge<HD, fa_sm103::one::kUnitRows1>(p, BH, N, stream);
  return FA_OK;
}

// Per-device facts, probed once: architecture and SM count.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return set_error(FA_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.probed) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_error("cudaDeviceGetAttribute", e);
    s.arch_ok = (major == 10 && minor == 3);
    s.num_sms = sms;
    s.probed = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn)
      return set_error(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = &s;
  return FA_OK;
}

// Range checks every entry point applies before any size arithmetic (B, H, N > 0, d a
// supported head dim): B*H, N and the work units fit the kernels' 32-bit indices, and
// the tensors' byte counts fit int64.
int check_ranges(int64_t B, int64_t H, int64_t N, int64_t d) {
  if (B > INT32_MAX / H) return set_error(FA_ERR_UNSUPPORTED, "B*H too large");
  const int64_t BH = B * H;
  if (N > (int64_t{1} << 30)) return set_error(FA_ERR_UNSUPPORTED, "N too large");
  // head dims 32 to 256 may run the one-tile kernel's 128-row units
  const int64_t unit_rows = d >= 32 ? fa_sm103::one::kUnitRows1 : fa_sm103::kUnitRows;
  if (((N + unit_rows - 1) / unit_rows) * BH > INT32_MAX)
    return set_error(FA_ERR_UNSUPPORTED, "too many work units");
  if (BH > (INT64_MAX / 4) / (N * d)) return set_error(FA_ERR_UNSUPPORTED, "tensor too large");
  return FA_OK;
}

// A launch's items (units x key-range pieces) index the kernels' schedule as int.
bool items_fit(int64_t BH, int64_t N, int kernel, int splits) {
  const int64_t rows = kernel == FA_KERNEL_ONE_TILE ? fa_sm103::one::kUnitRows1 : fa_sm103::kUnitRows;
  return ((N + rows - 1) / rows) * BH * splits <= INT32_MAX;
}

}  // namespace

namespace {

// Shared body of every forward entry point.  splits = 0 lets plan_for choose the kernel
// and the split count (among the counts the workspace holds); splits >= 1 runs that many
// pieces on `kernel`, or, when that is FA_KERNEL_AUTO, unsplit on the kernel plan_for
// picks and split on the two-tile kernel (the one-tile kernel at head dim 256).
int forward(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
            int64_t H, int64_t N, int64_t d, int causal, float scale, void* stream,
            const fa_fwd_options* opts, int splits, void* workspace, size_t workspace_size,
            int kernel = FA_KERNEL_AUTO) {
  t_last_error.clear();
  // ---- pure argument checks: no CUDA call before these pass ----
  if (B < 0 || H < 0 || N < 0) return set_error(FA_ERR_INVALID_ARG, "negative size");
  const int hd = head_dim_index(d);
  if (hd < 0) return set_error(FA_ERR_UNSUPPORTED, "head dim must be 16, 32, 64, 128 or 256");
  if (B == 0 || H == 0 || N == 0) return FA_OK;  // nothing to compute
  if (!q || !k || !v || !o) return set_error(FA_ERR_INVALID_ARG, "null tensor pointer");
  if (!std::isfinite(scale) || scale < 0.f)
    return set_error(FA_ERR_INVALID_ARG, "scale must be finite and >= 0");
  int st = check_ranges(B, H, N, d);
  if (st != FA_OK) return st;
  const int64_t BH = B * H;
  const size_t bytes = static_cast<size_t>(BH * N * d) * 2;
  const size_t lse_bytes = static_cast<size_t>(BH * N) * 4;
  for (const void* ptr : {q, k, v, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return set_error(FA_ERR_MISALIGNED, "tensor base address not 16-byte aligned");
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return set_error(FA_ERR_MISALIGNED, "lse not 4-byte aligned");
  for (const void* in : {q, k, v}) {
    if (overlaps(o, bytes, in, bytes)) return set_error(FA_ERR_INVALID_ARG, "o overlaps an input");
    if (lse && overlaps(lse, lse_bytes, in, bytes))
      return set_error(FA_ERR_INVALID_ARG, "lse overlaps an input");
  }
  if (lse && overlaps(lse, lse_bytes, o, bytes)) return set_error(FA_ERR_INVALID_ARG, "lse overlaps o");
  if (opts && (opts->wait_budget_cycles < 0 || opts->inject_skip_kv_load < 0 || opts->max_ctas < 0))
    return set_error(FA_ERR_INVALID_ARG, "negative option");
  if (opts && (opts->order < FA_ORDER_AUTO || opts->order > FA_ORDER_SHIFTED_SNAKES))
    return set_error(FA_ERR_INVALID_ARG, "unknown item order");
  const int block_kv = (opts && opts->block_kv != 0) ? opts->block_kv : 128;
  if (block_kv != 64 && block_kv != 128)
    return set_error(FA_ERR_INVALID_ARG, "block_kv must be 0 (automatic), 64 or 128");
  if (block_kv == 64) {  // 64-key tiles: the two-tile kernel only
    if (d == 256 || kernel == FA_KERNEL_ONE_TILE)
      return set_error(FA_ERR_UNSUPPORTED, "64-key tiles run on the two-tile kernel (head dims 16 to 128)");
    kernel = FA_KERNEL_TWO_TILE;
  }
  if (kernel < FA_KERNEL_AUTO || kernel > FA_KERNEL_ONE_TILE)
    return set_error(FA_ERR_INVALID_ARG, "unknown kernel");
  if (kernel == FA_KERNEL_TWO_TILE && d == 256)
    return set_error(FA_ERR_UNSUPPORTED, "the two-tile kernel serves head dims 16 to 128");
  if (kernel == FA_KERNEL_ONE_TILE && d < 32)
    return set_error(FA_ERR_UNSUPPORTED, "the one-tile kernel serves head dims 32 to 256");
  if (splits < 0 || splits > kMaxSplits)
    return set_error(FA_ERR_INVALID_ARG, "splits must be in [0, 64]");
  if (splits > 1 || (splits == 0 && workspace)) {
    if (!workspace) return set_error(FA_ERR_INVALID_ARG, "a split launch needs a workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
      return set_error(FA_ERR_MISALIGNED, "workspace not 16-byte aligned");
  }
  if (splits > 1 && !workspace_fits(workspace, workspace_size, BH, N, d, splits, q, k, v, o,
                                    bytes, lse, lse_bytes))
    return FA_ERR_INVALID_ARG;

  // ---- device checks ----
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != FA_OK) return st;
  if (!dev->arch_ok) return set_error(FA_ERR_ARCH, "device is not sm_103 (GB300-class)");
  if (splits == 0 && block_kv == 64) {
    // the two-tile kernel, split as the heuristic says (within the workspace given)
    const int max_splits =
        workspace ? splits_fitting(BH, N, d, static_cast<int64_t>(workspace_size)) : 1;
    splits = std::min(choose_splits(BH, N, dev->num_sms, causal), max_splits);
    if (splits > 1 && !workspace_fits(workspace, workspace_size, BH, N, d, splits, q, k, v, o,
                                      bytes, lse, lse_bytes))
      return FA_ERR_INVALID_ARG;
  } else if (splits == 0) {
    // plan among the split counts the workspace can hold
    const int max_splits =
        workspace ? splits_fitting(BH, N, d, static_cast<int64_t>(workspace_size)) : 1;
    const Plan pl = plan_cached(BH, N, d, causal, dev->num_sms, max_splits);
    kernel = pl.kernel;
    splits = pl.splits;
    if (splits > 1 && !workspace_fits(workspace, workspace_size, BH, N, d, splits, q, k, v, o,
                                      bytes, lse, lse_bytes))
      return FA_ERR_INVALID_ARG;
  } else if (kernel == FA_KERNEL_AUTO) {
    // unsplit: the planner's kernel; split as asked: the two-tile kernel (the one-tile
    // kernel at head dim 256, which the two-tile kernel does not serve)
    kernel = splits == 1 ? plan_cached(BH, N, d, causal, dev->num_sms, 1).kernel
             : d == 256  ? static_cast<int>(FA_KERNEL_ONE_TILE)
                         : static_cast<int>(FA_KERNEL_TWO_TILE);
  }
  if (!items_fit(BH, N, kernel, splits))
    return set_error(FA_ERR_UNSUPPORTED, "too many work items (units x splits)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kernel == FA_KERNEL_ONE_TILE) {
    bool& set_one = dev->smem_set_one[hd];
    switch (hd) {
      case 1: return launch_one<32>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, set_one, opts, splits, workspace);
      case 2: return launch_one<64>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, set_one, opts, splits, workspace);
      case 3: return launch_one<128>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, set_one, opts, splits, workspace);
      default: return launch_one<256>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, set_one, opts, splits, workspace);
    }
  }
  bool& smem_set = dev->smem_set[hd][block_kv == 64 ? 1 : 0];
  if (block_kv == 64) {
    switch (hd) {
      case 0: return launch<16, 64>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
      case 1: return launch<32, 64>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
      case 2: return launch<64, 64>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
      default: return launch<128, 64>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
    }
  }
  switch (hd) {
    case 0: return launch<16, 128>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
    case 1: return launch<32, 128>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
    case 2: return launch<64, 128>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
    default: return launch<128, 128>(q, k, v, o, lse, BH, N, causal, scale, s, *dev, smem_set, opts, splits, workspace);
  }
}

}  // namespace

extern "C" {

int fa_fwd_opts(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                int64_t H, int64_t N, int64_t d, int causal, float scale, void* stream,
                const fa_fwd_options* opts) {
  return forward(q, k, v, o, lse, B, H, N, d, causal, scale, stream, opts, 1, nullptr, 0,
                 opts ? opts->kernel : FA_KERNEL_AUTO);
}

int64_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int splits) {
  if (B < 0 || H < 0 || N < 0 || head_dim_index(d) < 0 || splits < 1 || splits > kMaxSplits)
    return -1;
  if (B == 0 || H == 0 || N == 0) return 0;
  if (check_ranges(B, H, N, d) != FA_OK) return -1;
  // the two-tile kernel's 256-row items are the larger count of rows; both kernels' items
  // must fit the schedule's int index
  if (!items_fit(B * H, N, FA_KERNEL_ONE_TILE, splits)) return -1;
  return workspace_bytes(B * H, N, d, splits);
}

int fa_splitkv_auto_splits(int64_t B, int64_t H, int64_t N, int causal) {
  if (B <= 0 || H <= 0 || N <= 0) return 1;
  DeviceState* dev = nullptr;
  if (device_state(&dev) != FA_OK) return 1;
  return choose_splits(B * H, N, dev->num_sms, causal);
}

int fa_fwd_plan(int64_t B, int64_t H, int64_t N, int64_t d, int causal, int allow_split,
                int num_sms, int* kernel, int* splits, int* order) {
  t_last_error.clear();
  if (!kernel || !splits) return set_error(FA_ERR_INVALID_ARG, "null output pointer");
  if (B < 0 || H < 0 || N < 0 || num_sms < 0) return set_error(FA_ERR_INVALID_ARG, "negative size");
  if (head_dim_index(d) < 0) return set_error(FA_ERR_UNSUPPORTED, "head dim must be 16, 32, 64, 128 or 256");
  if (B == 0 || H == 0 || N == 0) {
    *kernel = d == 256 ? FA_KERNEL_ONE_TILE : FA_KERNEL_TWO_TILE;
    *splits = 1;
    if (order) *order = FA_ORDER_ONE_SNAKE;
    return FA_OK;
  }
  if (B > INT32_MAX / H || N > (int64_t{1} << 30))
    return set_error(FA_ERR_UNSUPPORTED, "sizes beyond the kernel's range");
  int sms = num_sms;
  if (sms == 0) {
    DeviceState* dev = nullptr;
    const int st = device_state(&dev);
    if (st != FA_OK) return st;
    sms = dev->num_sms;
  }
  const Plan pl = plan_cached(B * H, N, d, causal ? 1 : 0, sms, allow_split ? kMaxSplits : 1);
  *kernel = pl.kernel;
  *splits = pl.splits;
  if (order) {
    const int64_t rows = pl.kernel == FA_KERNEL_ONE_TILE ? fa_sm103::one::kUnitRows1 : fa_sm103::kUnitRows;
    const int64_t items = (N + rows - 1) / rows * B * H * pl.splits;
    const int grid = static_cast<int>(std::min<int64_t>(sms, items));
    const int o = schedule_order(pl.kernel, B * H, N, d, causal, grid, pl.splits);
    *order = o == 1 ? FA_ORDER_GROUP_SNAKES : o == 2 ? FA_ORDER_SHIFTED_SNAKES : FA_ORDER_ONE_SNAKE;
  }
  return FA_OK;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                   int64_t H, int64_t N, int64_t d, int causal, float scale, int splits,
                   void* workspace, size_t workspace_bytes_given, void* stream) {
  return forward(q, k, v, o, lse, B, H, N, d, causal, scale, stream, nullptr, splits, workspace,
                 workspace_bytes_given);
}

int fa_fwd_splitkv_opts(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                        int splits, void* workspace, size_t workspace_bytes_given, void* stream,
                        const fa_fwd_options* opts) {
  const int kernel = opts ? opts->kernel : FA_KERNEL_AUTO;
  if (splits == 0 && kernel != FA_KERNEL_AUTO) {
    t_last_error.clear();
    return set_error(FA_ERR_INVALID_ARG, "a pinned kernel needs an explicit split count");
  }
  return forward(q, k, v, o, lse, B, H, N, d, causal, scale, stream, opts, splits, workspace,
                 workspace_bytes_given, kernel);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
           int64_t N, int64_t d, int causal, float scale, void* stream) {
  return fa_fwd_opts(q, k, v, o, lse, B, H, N, d, causal, scale, stream, nullptr);
}

}  // extern "C"

namespace {

// Device address of g_static_scratch on the current device.  In host code the array's
// name is only a stand-in, so the address is asked for once per device (with that
// device current) and kept.
void* g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];

int static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return set_error(FA_ERR_UNSUPPORTED, "device index too large");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ready[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_error("cudaGetSymbolAddress(static scratch)", e);
    g_scratch_ptr[dev] = ptr;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                           int splits, void* stream) {
  t_last_error.clear();
  if (B < 0 || H < 0 || N < 0) return set_error(FA_ERR_INVALID_ARG, "negative size");
  if (head_dim_index(d) < 0) return set_error(FA_ERR_UNSUPPORTED, "head dim must be 16, 32, 64, 128 or 256");
  if (splits < 0 || splits > kMaxSplits) return set_error(FA_ERR_INVALID_ARG, "splits must be in [0, 64]");
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  int st = check_ranges(B, H, N, d);
  if (st != FA_OK) return st;
  if (splits > 1 && !items_fit(B * H, N, FA_KERNEL_ONE_TILE, splits))
    return set_error(FA_ERR_UNSUPPORTED, "too many work items (units x splits)");
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != FA_OK) return st;
  int kernel = FA_KERNEL_AUTO;
  if (splits == 0) {
    const Plan pl = plan_cached(B * H, N, d, causal ? 1 : 0, dev->num_sms,
                                splits_fitting(B * H, N, d, static_cast<int64_t>(kStaticScratchBytes)));
    kernel = pl.kernel;
    splits = pl.splits;
  }
  const int64_t need = workspace_bytes(B * H, N, d, splits);
  if (need > static_cast<int64_t>(kStaticScratchBytes)) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "needs %lld bytes of scratch but the built-in scratch holds %zu (64 MiB); use "
             "fa_fwd_splitkv with a workspace, or fewer splits",
             static_cast<long long>(need), kStaticScratchBytes);
    return set_error(FA_ERR_UNSUPPORTED, buf);
  }
  void* scratch = nullptr;
  if (splits > 1 && (st = static_scratch_address(&scratch)) != FA_OK) return st;
  return forward(q, k, v, o, lse, B, H, N, d, causal, scale, stream, nullptr, splits, scratch,
                 splits > 1 ? kStaticScratchBytes : 0, kernel);
}

int64_t fa_noalloc_scratch_bytes(void) { return static_cast<int64_t>(kStaticScratchBytes); }

}  // extern "C"

extern "C" {

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported size or head dimension";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_ARCH: return "device is not sm_103";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel wait ran out of time";
    default: return "unknown status";
  }
}

const char* fa_last_error(void) { return t_last_error.c_str(); }

int fa_get_device_status(void* stream) {
  t_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error("cudaStreamSynchronize", e);
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, fa_sm103::g_device_status, sizeof word);
  if (e != cudaSuccess) return cuda_error("cudaMemcpyFromSymbol", e);
  if (word == 0) return FA_OK;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(fa_sm103::g_device_status, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_error("cudaMemcpyToSymbol", e);
  return FA_ERR_DEVICE_TIMEOUT;
}

int fa_version(void) { return kVersion; }

int fa_row_kernel_register_check(int num_regs, int max_threads_per_block) {
  t_last_error.clear();
  return register_split_check(num_regs, max_threads_per_block);
}

void fa_test_override_kernel_registers(int num_regs) {
  g_regs_override.store(num_regs > 0 ? num_regs : 0);
}

}  // extern "C"
