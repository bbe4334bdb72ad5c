// api.cu - host side of the C ABI: plan (validation, bucketing, cost-ordered
// tile lists, workspace layout), bind (tables and TMA tensor maps), step
// (the launch sequence), profiling and introspection.
//
// Batching: matrices with the same (short, long) shape form one bucket, laid
// out as a [count, m, ld] array in the workspace; every phase of the
// Newton-Schulz iteration then runs the tiles of all buckets in one launch
// ("DMuon: Efficient Distributed Muon Training with Near-Adam Overhead",
// gist.science summary section 2, "Batching": batch matrices of similar shape
// and run the recurrence jointly to amortise dispatch). Within a launch the
// tiles are sorted by cost, largest first, and each persistent CTA (or CTA
// pair) claims the next one from a counter when it becomes free: list
// scheduling in cost order, the greedy makespan balancing of section 2.3
// applied to SMs instead of owner ranks (DMUON_FLAG_STATIC_TILES deals the
// same list round-robin instead).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <string>
#include <vector>

#include "dmuon.h"
#include "internal.h"
#include "simt.h"

using namespace dmuon;

namespace {

thread_local std::string g_err;

// DMUON_LOG=1 in the environment: the library writes one line per plan, bind,
// first step of a plan and error to stderr. Otherwise it writes nothing.
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("DMUON_LOG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

void logf(const char* fmt, ...) {
  if (!log_enabled()) return;
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  std::fprintf(stderr, "[dmuon] %s\n", buf);
}

dmuon_status fail(dmuon_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  logf("error %d: %s", static_cast<int>(st), buf);
  return st;
}

// NVTX range names per launch kind (host-side ranges around each launch of a
// step; free when no profiling tool is attached).
const char* kind_range_name(int kind) {
  switch (kind) {
    case DMUON_KIND_MOMENTUM: return "dmuon momentum";
    case DMUON_KIND_GRAM: return "dmuon gram X X^T";
    case DMUON_KIND_POLY: return "dmuon poly aI + bA + cA^2";
    case DMUON_KIND_GEMM: return "dmuon gemm P X";
    case DMUON_KIND_UPDATE0: return "dmuon update (ns_steps 0)";
    case DMUON_KIND_SYMM: return "dmuon symm (Gram form)";
    case DMUON_KIND_NORM: return "dmuon norm";
    default: return "dmuon launch";
  }
}

dmuon_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DMUON_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kAlign = 1024;
constexpr int64_t kProbeTiles = 4096;  // tile-list room of one tuning probe
constexpr int64_t kSchedBytes = 128;   // one launch's tile-claim counters (own cache line)
int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kPtrSlots = 4;  // device-resident pointer tables per plan

// Host-side failure injection for tests: true when the environment variable
// DMUON_TEST_FAIL names this point of dmuon_plan_bind. Nothing on the device
// is involved; the call then fails as if the CUDA call at that point had.
bool test_hook(const char* where) {
  const char* v = std::getenv("DMUON_TEST_FAIL");
  return v != nullptr && std::strcmp(v, where) == 0;
}

// Test hook: true when the environment variable `name` is set to a non-empty value other than "0".
// DMUON_TEST_FORCE_PAIRS with DMUON_FLAG_PAIR_TILES gives every bucket with a short side >= 256
// two-SM pair tiles (as tuning may), also where the short side is not a multiple of 256.
bool test_hook_env(const char* name) {
  const char* v = std::getenv(name);
  return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
}

// Test hook of the debug checks: DMUON_TEST_SKIP_LAUNCH=<i> leaves launch i of
// every step out (only under DMUON_FLAG_DEBUG_CHECKS), so that its outputs are
// stale and the checks must report them.
bool test_skip_launch(int li) {
  const char* v = std::getenv("DMUON_TEST_SKIP_LAUNCH");
  return v != nullptr && v[0] != '\0' && std::atoi(v) == li;
}

// Workspace buffers of a bucket, by role. Standard buckets use X0/X1 (the
// iterate, ping-pong), A and B; Gram-space buckets use X0 (U, read twice), G,
// P, Q0/Q1 (ping-pong) and R.
enum BufRole : int { kBufNone = -1, kBufX0 = 0, kBufX1, kBufA, kBufB, kBufQ0, kBufQ1, kBufR, kBufCount };

struct BucketPlan {
  int32_t m = 0, n = 0, count = 0, n_transposed = 0;
  int32_t x_ld = 0, m_ld = 0;
  bool gram = false;          // iterate in the m x m Gram space
  bool pair = false;          // 256 x 256 tiles on CTA pairs (two-SM UMMA)
  int32_t bn_sym = 0;         // tile width of the symmetric products (m x m outputs)
  int32_t bn_gemm = 0;        // tile width of the m x n product
  // measured SM-ms per tile (time per tile x SMs it occupies): X X^T (K = n), m x m products, gemm;
  // 0 = not measured
  double tile_ms[3] = {0, 0, 0};
  double tune_cost[3] = {0, 0, 0};  // tuning: SM-ms per matrix of one-SM 128, one-SM 256, pairs (0 = not timed)
  double tune_gemm[3] = {0, 0, 0};  // the part of tune_cost spent in the gemm
  std::vector<int32_t> mats;  // slot -> global matrix index
  int64_t off_slotmat = -1;
  int64_t off[kBufCount] = {-1, -1, -1, -1, -1, -1, -1};
  int64_t x_mat_bytes = 0, a_mat_bytes = 0;
  bool is_x(int role) const { return role == kBufX0 || role == kBufX1; }
};

struct ListRef {
  int64_t first = 0;  // index into items
  int32_t count = 0;
};

enum ListKind : int { kListGram = 0, kListPoly = 1, kListGemm = 2 };

struct Launch {
  int kind = 0;   // DMUON_KIND_*
  int phase = 0;  // kernel: kPhaseGram / kPhasePoly / kPhaseGemm
  int step = -1;  // Newton-Schulz step
  int chunk = 0;
  int list = 0;   // ListKind
  int bn = 0;     // tile width of this launch
  bool pair = false;  // two-SM tiles
  int opA = kBufNone, opB = kBufNone, out = kBufNone, aux = kBufNone;
  float a = 0.f, b = 0.f, c = 0.f, diag = 0.f;
  int first = 0, last = 0;
  int32_t grid = 0;
  double work = 0;  // algorithmic flops (products) or bytes (streaming)
  int param_index = -1;
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

struct dmuon_plan_s {
  // ---- description
  std::vector<dmuon_shape> shapes;
  int32_t ns_steps = 0;
  std::vector<float> coeffs;  // 3 * ns_steps
  float eps = 0.f;
  dmuon_dtypes dt{};
  uint32_t flags = 0;
  bool tc = false;  // bf16 compute: tensor-core path
  int xel = 4;      // workspace element size
  int tile_m = 0, tile_n = 0;
  // ---- derived
  std::vector<MatDev> mats;
  std::vector<int64_t> unit_begin;
  int64_t n_units = 0;
  std::vector<BucketPlan> buckets;
  std::vector<std::vector<int>> chunks;
  std::vector<bool> chunk_gram;
  std::vector<int4> items;
  std::vector<ListRef> gram_lists, poly_lists, gemm_lists;
  std::vector<Launch> launches;
  // ---- workspace layout (byte offsets)
  size_t ws_bytes = 0;
  int64_t off_status = 0, off_s = 0, off_partial = 0, off_mats = 0, off_ub = 0, off_ptrs = 0,
          off_items = 0, off_probe = 0, off_capture = -1, off_wmaps = -1, off_sched = 0, off_cta = 0,
          off_probe_sched = 0;
  int64_t cap_elems = 0;
  // ---- binding
  char* ws = nullptr;
  int device = -1;
  int num_sms = 0;
  StreamParams sp{};
  std::vector<TcParams> tc_params;
  std::vector<SimtParams> simt_params;
  // Device-resident pointer tables (W, G, M device pointers per matrix), kPtrSlots of them, so
  // that a step whose pointers match a resident table uploads nothing: alternating gradient
  // buffers cost no copy after the first step with each. Each slot has its own pinned staging
  // and an event that guards that staging until its upload has read it.
  uint64_t* host_ptrs = nullptr;  // pinned staging, kPtrSlots tables
  // With each resident pointer set, a TMA map of every W (tensor-core path, bf16 weights): the
  // last step's epilogue stores its updated W boxes through them. Pinned staging per slot.
  CUtensorMap* host_wmaps = nullptr;
  // mapped page-locked word that dmuon_read_device_status reads the status into (host and device
  // addresses)
  unsigned* host_status = nullptr;
  unsigned* host_status_dev = nullptr;
  std::vector<uint64_t> slot_ptrs[kPtrSlots];
  uint64_t slot_stamp[kPtrSlots] = {};
  uint64_t ptr_clock = 0;
  cudaEvent_t ptr_event[kPtrSlots] = {};
  bool ptr_event_pending[kPtrSlots] = {};
  // ---- profiling
  bool prof = false;
  int32_t prof_max = 0, prof_n = 0;
  std::vector<cudaEvent_t> ev_start, ev_stop;
  std::vector<int32_t> prof_kind;
  std::vector<double> prof_work;
  int64_t launch_count = 0;
  int64_t steps_taken = 0;
  bool tuned = false;
  int tune_timed = 0, tune_cached = 0;  // buckets timed at bind / taken from the tuning cache
  bool cta_times = false;  // dmuon_profile_cta_times: record per-CTA start/end of tensor-core launches
  // ---- ordering of the weight writes against other streams (dmuon_set_weight_events)
  cudaEvent_t w_wait = nullptr;   // waited on before the first launch that writes W
  cudaEvent_t w_done = nullptr;   // recorded after the last launch that writes W
  int first_w_launch = -1, last_w_launch = -1;  // indices into launches
};

namespace {

double phase_flops(int kind, double m, double n) {
  switch (kind) {
    case DMUON_KIND_GRAM:
      return m * (m + 1) * n;
    case DMUON_KIND_POLY:
    case DMUON_KIND_SYMM:
      return m * m * (m + 1);
    case DMUON_KIND_GEMM:
      return 2 * m * m * n;
    default:
      return 0;
  }
}

int dtype_bytes(int32_t d) { return d == DMUON_BF16 ? 2 : 4; }

// Default tile widths. A 128 x 256 tile takes about 1.4x the time of a 128 x 128
// one over the same K (it moves 48 KB of operands per 64-wide K slice against
// 32 KB, for twice the flops; timed on the 1408-row MoE experts: the symmetric
// products ran 66 tiles of 128 in 78 ms and 41 tiles of 256 in 66 ms). So 256
// is the default unless its tiles, weighted by 1.4, outnumber those of 128.
constexpr double kWideTileCost = 1.4;

// Shortest short side that gets two-SM pair tiles by default.
constexpr int kPairMinShort = 1024;

// Tiles of a symmetric m x m product: row block ti (bm rows) covers columns
// from its diagonal block on, ti*bm + tj*bn for tj = 0, 1, ..., so no tile
// reaches below the diagonal block of its rows.
int64_t sym_tiles(int m, int bm, int bn) {
  int64_t t = 0;
  for (int64_t ti = 0; ti < cdiv(m, bm); ++ti) t += cdiv(m - ti * bm, bn);
  return t;
}

int32_t default_bn_sym(int m) {
  return kWideTileCost * sym_tiles(m, kTcBM, 256) <= sym_tiles(m, kTcBM, 128) ? 256 : 128;
}
int32_t default_bn_gemm(int n) { return kWideTileCost * cdiv(n, 256) <= cdiv(n, 128) ? 256 : 128; }

// Tiles of one phase for one bucket, appended in cost order.
void add_tiles(const dmuon_plan_s& P, int kind, int bucket_local, const BucketPlan& B, std::vector<int4>& out) {
  const int BM = B.pair ? 256 : P.tile_m, BN = (kind == DMUON_KIND_GEMM) ? B.bn_gemm : B.bn_sym;
  const int tm = static_cast<int>(cdiv(B.m, BM));
  if (kind == DMUON_KIND_GEMM) {
    const int tn = static_cast<int>(cdiv(B.n, BN));
    for (int s = 0; s < B.count; ++s)
      for (int tj = 0; tj < tn; ++tj)
        for (int ti = 0; ti < tm; ++ti) out.push_back(make_int4(bucket_local, s, ti, tj));
  } else {  // symmetric products: tile (ti, tj) covers columns ti*BM + tj*BN.. (from the diagonal block on)
    for (int s = 0; s < B.count; ++s)
      for (int ti = 0; ti < tm; ++ti)
        for (int tj = 0; tj < static_cast<int>(cdiv(B.m - ti * BM, BN)); ++tj)
          out.push_back(make_int4(bucket_local, s, ti, tj));
  }
}

dmuon_status finish_plan(dmuon_plan_s& P);

// Buckets (with default tile widths), per-matrix tables and streaming units.
dmuon_status build_plan(dmuon_plan_s& P) {
  const int n_mats = static_cast<int>(P.shapes.size());
  P.tc = (P.dt.compute == DMUON_BF16);
  P.xel = P.tc ? 2 : 4;
  P.tile_m = P.tc ? kTcBM : kSimtBM;
  P.tile_n = P.tc ? kTcBN : kSimtBN;
  // Row pitch of the m x n iterates: tensor-core buckets round n up to 64 elements, so that the
  // gemm's 4-D view of X (64-column chunks of a row) never reads past a row; m x m buffers and the
  // fp32 path round to 16 bytes (TMA strides)
  const int ld_mult = P.tc ? 64 : 4;
  const int m_ld_mult = P.tc ? 8 : 4;

  // ---- buckets by (short, long) shape, most expensive first
  std::map<std::pair<int, int>, int> key;
  std::vector<std::pair<int, int>> order;
  for (int i = 0; i < n_mats; ++i) {
    const int r = static_cast<int>(P.shapes[i].rows), c = static_cast<int>(P.shapes[i].cols);
    const std::pair<int, int> k{std::min(r, c), std::max(r, c)};
    if (!key.count(k)) {
      key[k] = 0;
      order.push_back(k);
    }
  }
  std::stable_sort(order.begin(), order.end(), [](auto a, auto b) {
    return 1.0 * a.first * a.first * a.second > 1.0 * b.first * b.first * b.second;
  });
  P.buckets.assign(order.size(), BucketPlan{});
  for (size_t b = 0; b < order.size(); ++b) {
    key[order[b]] = static_cast<int>(b);
    P.buckets[b].m = order[b].first;
    P.buckets[b].n = order[b].second;
    P.buckets[b].x_ld = static_cast<int32_t>(align_up(order[b].second, ld_mult));
    P.buckets[b].m_ld = static_cast<int32_t>(align_up(order[b].first, m_ld_mult));
    // the Gram-space form pays (>= 26% fewer flops) and keeps bf16 accuracy on wide matrices only
    P.buckets[b].gram = (P.flags & DMUON_FLAG_GRAM_NS) && P.ns_steps >= 1 && order[b].second >= 2 * order[b].first;
    P.buckets[b].bn_sym = P.tc ? default_bn_sym(order[b].first) : kSimtBN;
    P.buckets[b].bn_gemm = P.tc ? default_bn_gemm(order[b].second) : kSimtBN;
    // two-SM 256 x 256 tiles (the default) where they fill the short side, so that no 256-row tile is
    // left half empty, and where it spans at least 4 row pairs: below that the diagonal pair tiles,
    // half of whose work lies below the diagonal, weigh too much (measured by tuning: short sides of
    // 256 and 512 run 9-12 % faster on one-SM tiles, 1024 level, 1536 and up faster on pairs).
    // DMUON_FLAG_PAIR_TILES asks for them on shorter sides too. Tuning may still choose pairs for
    // other short sides >= 256, and so does the test hook.
    const bool pairs_on = P.tc && !(P.flags & DMUON_FLAG_ONE_SM_TILES);
    const bool forced = pairs_on && order[b].first >= 256 && test_hook_env("DMUON_TEST_FORCE_PAIRS");
    const bool long_enough = order[b].first >= kPairMinShort || (P.flags & DMUON_FLAG_PAIR_TILES);
    if (forced) P.buckets[b].bn_sym = P.buckets[b].bn_gemm = 256;
    P.buckets[b].pair = forced || (pairs_on && order[b].first % 256 == 0 && long_enough &&
                                   P.buckets[b].bn_sym == 256 && P.buckets[b].bn_gemm == 256);
  }

  P.mats.assign(n_mats, MatDev{});
  P.unit_begin.assign(n_mats + 1, 0);
  int64_t units = 0, cap = 0;
  for (int i = 0; i < n_mats; ++i) {
    const int r = static_cast<int>(P.shapes[i].rows), c = static_cast<int>(P.shapes[i].cols);
    MatDev& d = P.mats[i];
    d.rows = r;
    d.cols = c;
    d.m = std::min(r, c);
    d.n = std::max(r, c);
    d.transposed = r > c;
    d.bucket = key[{d.m, d.n}];
    BucketPlan& B = P.buckets[d.bucket];
    d.slot = B.count++;
    B.mats.push_back(i);
    B.n_transposed += d.transposed;
    d.x_ld = B.x_ld;
    d.scale = static_cast<float>(std::sqrt(std::max(1.0, static_cast<double>(r) / c)));
    d.flat = (!d.transposed && c % 8 == 0 && d.x_ld == c) ? 1 : 0;  // U rows land contiguous
    d.tiles_c = static_cast<int32_t>(cdiv(c, kTileC));
    d.vec_ok = (c % 4 == 0) ? 1 : 0;
    d.unit_begin = units;
    d.unit_count = d.flat ? cdiv((int64_t)r * c, kFlatUnit) : cdiv(r, kTileR) * cdiv(c, kTileC);
    units += d.unit_count;
    P.unit_begin[i] = d.unit_begin;
    if (P.flags & DMUON_FLAG_CAPTURE_UPDATE) {
      d.cap_off = cap;
      cap += align_up((int64_t)r * c, 64);
    } else {
      d.cap_off = -1;
    }
  }
  P.unit_begin[n_mats] = units;
  P.n_units = units;
  P.cap_elems = cap;
  return finish_plan(P);
}

// Tile widths, launch chunks, cost-ordered tile lists, workspace layout and
// launch sequence. Called again after tuning changes tile widths or costs;
// the workspace layout does not move (the tile-list region is sized for the
// largest possible lists).
dmuon_status finish_plan(dmuon_plan_s& P) {
  const int n_mats = static_cast<int>(P.shapes.size());
  const int64_t units = P.n_units, cap = P.cap_elems;

  // ---- launch chunks: at most kMaxBucketsPerLaunch buckets sharing iteration form and tile widths
  P.chunks.clear();
  P.chunk_gram.clear();
  {
    std::vector<std::tuple<int, int, int, int>> keys;
    for (const BucketPlan& B : P.buckets) {
      const auto k = std::make_tuple((int)B.gram, B.bn_sym, B.bn_gemm, (int)B.pair);
      if (std::find(keys.begin(), keys.end(), k) == keys.end()) keys.push_back(k);
    }
    std::stable_sort(keys.begin(), keys.end(),
                     [](const auto& a, const auto& b) { return std::get<0>(a) < std::get<0>(b); });
    for (const auto& k : keys) {
      std::vector<int> ch;
      for (size_t b = 0; b < P.buckets.size(); ++b) {
        const BucketPlan& B = P.buckets[b];
        if (std::make_tuple((int)B.gram, B.bn_sym, B.bn_gemm, (int)B.pair) != k) continue;
        ch.push_back(static_cast<int>(b));
        if (ch.size() == kMaxBucketsPerLaunch) {
          P.chunks.push_back(ch);
          P.chunk_gram.push_back(std::get<0>(k) != 0);
          ch.clear();
        }
      }
      if (!ch.empty()) {
        P.chunks.push_back(ch);
        P.chunk_gram.push_back(std::get<0>(k) != 0);
      }
    }
  }

  // ---- cost-ordered tile lists per (phase, chunk)
  P.items.clear();
  auto build_list = [&](int kind, const std::vector<int>& ch) {
    std::vector<std::pair<double, int4>> tmp;
    for (size_t lb = 0; lb < ch.size(); ++lb) {
      const BucketPlan& B = P.buckets[ch[lb]];
      std::vector<int4> t;
      add_tiles(P, kind, static_cast<int>(lb), B, t);
      // cost of one tile: its measured time when the plan was tuned, else its K extent
      const int li = (kind == DMUON_KIND_GRAM) ? 0 : (kind == DMUON_KIND_POLY) ? 1 : 2;
      const double cost = B.tile_ms[li] > 0 ? B.tile_ms[li] * 1e9 : (kind == DMUON_KIND_GRAM) ? B.n : B.m;
      for (const int4& v : t) tmp.push_back({cost, v});
    }
    std::stable_sort(tmp.begin(), tmp.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
    ListRef ref;
    ref.first = static_cast<int64_t>(P.items.size());
    ref.count = static_cast<int32_t>(tmp.size());
    for (auto& v : tmp) P.items.push_back(v.second);
    return ref;
  };
  P.gram_lists.clear();
  P.poly_lists.clear();
  P.gemm_lists.clear();
  if (P.ns_steps > 0) {
    for (const auto& ch : P.chunks) {
      P.gram_lists.push_back(build_list(DMUON_KIND_GRAM, ch));
      P.poly_lists.push_back(build_list(DMUON_KIND_POLY, ch));
      P.gemm_lists.push_back(build_list(DMUON_KIND_GEMM, ch));
    }
  }

  // ---- workspace layout
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = align_up(off + std::max<int64_t>(bytes, 1), kAlign);
    return o;
  };
  P.off_status = take(256);
  P.off_s = take(4LL * n_mats);
  P.off_partial = take(4LL * kPartialsPerUnit * std::max<int64_t>(units, 1));
  P.off_mats = take((int64_t)sizeof(MatDev) * n_mats);
  P.off_ub = take(8LL * (n_mats + 1));
  P.off_ptrs = take(8LL * 3 * n_mats * kPtrSlots);
  if (P.tc && P.dt.param == DMUON_BF16 && P.ns_steps > 0)
    P.off_wmaps = take((int64_t)sizeof(CUtensorMap) * n_mats * kPtrSlots);
  // tile lists: room for the longest lists any choice of tile widths gives (all 128 wide)
  int64_t cap_items = 0;
  if (P.ns_steps > 0) {
    for (const BucketPlan& B : P.buckets) {
      const int64_t tm = cdiv(B.m, P.tile_m), bn = P.tc ? 128 : kSimtBN;
      cap_items += B.count * (2 * sym_tiles(B.m, P.tile_m, static_cast<int>(bn)) + tm * cdiv(B.n, bn));
    }
  }
  P.off_items = take((int64_t)sizeof(int4) * std::max<int64_t>(std::max<int64_t>(cap_items, (int64_t)P.items.size()), 1));
  P.off_probe = take((int64_t)sizeof(int4) * kProbeTiles);
  // per launch of a step (and one for the tuning probes): the tile-claim counter pair, 128 bytes
  // apart; and the per-CTA profiling records of each launch. The launch count is bounded by the
  // step's sequence below, 3 + 4 * ns_steps per launch chunk at most, and a chunk holds at least one
  // bucket. The bound uses the bucket count, which tuning does not change (it may split buckets
  // into more chunks): the layout of the workspace must not move when tuning re-plans.
  const int64_t max_launches = 3 + 4LL * std::max(P.ns_steps, 1) * std::max<int64_t>((int64_t)P.buckets.size(), 1);
  P.off_sched = take(kSchedBytes * (max_launches + 1));
  P.off_probe_sched = P.off_sched + kSchedBytes * max_launches;
  P.off_cta = take(16LL * kMaxCtaRecords * max_launches);
  for (BucketPlan& B : P.buckets) {
    B.off_slotmat = take(4LL * B.count);
    B.x_mat_bytes = (int64_t)B.m * B.x_ld * P.xel;
    B.a_mat_bytes = (int64_t)B.m * B.m_ld * P.xel;
    B.off[kBufX0] = take(B.x_mat_bytes * B.count);
    if (!B.gram) {
      if (P.ns_steps >= 2) B.off[kBufX1] = take(B.x_mat_bytes * B.count);
      if (P.ns_steps >= 1) {
        B.off[kBufA] = take(B.a_mat_bytes * B.count);
        B.off[kBufB] = take(B.a_mat_bytes * B.count);
      }
    } else {
      B.off[kBufA] = take(B.a_mat_bytes * B.count);   // G
      B.off[kBufQ0] = take(B.a_mat_bytes * B.count);  // P_0 = Q_1, then every other Q
      if (P.ns_steps >= 2) {
        B.off[kBufB] = take(B.a_mat_bytes * B.count);   // P_k, k >= 1
        B.off[kBufQ1] = take(B.a_mat_bytes * B.count);
        B.off[kBufR] = take(B.a_mat_bytes * B.count);   // P_k G_k
      }
    }
  }
  for (int i = 0; i < n_mats; ++i) {
    const BucketPlan& B = P.buckets[P.mats[i].bucket];
    P.mats[i].x0_off = B.off[kBufX0] + (int64_t)P.mats[i].slot * B.x_mat_bytes;
  }
  P.off_capture = (P.flags & DMUON_FLAG_CAPTURE_UPDATE) ? take(4 * std::max<int64_t>(cap, 1)) : -1;
  P.ws_bytes = static_cast<size_t>(off);

  // ---- launch sequence (grid sizes are filled in at bind, when the SM count is known)
  P.launches.clear();
  const int gb = dtype_bytes(P.dt.grad), pb = dtype_bytes(P.dt.param);
  double elems = 0;
  for (const auto& s : P.shapes) elems += static_cast<double>(s.rows) * s.cols;
  Launch L;
  L.kind = DMUON_KIND_MOMENTUM;
  L.work = elems * (gb + 4 + 4 + P.xel);
  P.launches.push_back(L);
  Launch nf;
  nf.kind = DMUON_KIND_NORM;
  nf.work = 4.0 * kPartialsPerUnit * static_cast<double>(P.n_units) + 4.0 * n_mats;  // partials read, s written
  P.launches.push_back(nf);
  if (P.ns_steps == 0) {
    Launch u;
    u.kind = DMUON_KIND_UPDATE0;
    u.work = elems * (2 * pb + P.xel);
    P.launches.push_back(u);
  }
  auto add = [&](int kind, int phase, int step, int chunk, int list, int opA, int opB, int out, int aux, float a,
                 float b, float c, float diag, int first, int last) {
    Launch x;
    x.kind = kind;
    x.phase = phase;
    x.step = step;
    x.chunk = chunk;
    x.list = list;
    x.bn = (phase == kPhaseGemm) ? P.buckets[P.chunks[chunk][0]].bn_gemm : P.buckets[P.chunks[chunk][0]].bn_sym;
    x.pair = P.buckets[P.chunks[chunk][0]].pair;
    x.opA = opA;
    x.opB = opB;
    x.out = out;
    x.aux = aux;
    x.a = a;
    x.b = b;
    x.c = c;
    x.diag = diag;
    x.first = first;
    x.last = last;
    for (int bi : P.chunks[chunk]) {
      const BucketPlan& B = P.buckets[bi];
      x.work += B.count * phase_flops(kind, B.m, B.n);
    }
    P.launches.push_back(x);
  };
  const int S = P.ns_steps;
  auto cf = [&](int k, int q) { return P.coeffs[3 * k + q]; };
  // standard form, step by step: A = X X^T; P = a I + b A + c A A^T; X' = P X (last: W update).
  // With DMUON_FLAG_EPILOGUE_AX: B = b A + c A A^T and X' = a X + B X, a*X read in the epilogue.
  const bool ax_epilogue = (P.flags & DMUON_FLAG_EPILOGUE_AX) != 0;
  for (int k = 0; k < S; ++k) {
    const int xin = (k & 1) ? kBufX1 : kBufX0, xout = (k & 1) ? kBufX0 : kBufX1;
    for (size_t ch = 0; ch < P.chunks.size(); ++ch)
      if (!P.chunk_gram[ch])
        add(DMUON_KIND_GRAM, kPhaseGram, k, (int)ch, kListGram, xin, xin, kBufA, kBufNone, 0, 0, 0, 0, k == 0, 0);
    for (size_t ch = 0; ch < P.chunks.size(); ++ch)
      if (!P.chunk_gram[ch])
        add(DMUON_KIND_POLY, kPhasePoly, k, (int)ch, kListPoly, kBufA, kBufA, kBufB, kBufA, 0, cf(k, 1), cf(k, 2),
            ax_epilogue ? 0.f : cf(k, 0), 0, 0);
    for (size_t ch = 0; ch < P.chunks.size(); ++ch)
      if (!P.chunk_gram[ch])
        add(DMUON_KIND_GEMM, kPhaseGemm, k, (int)ch, kListGemm, kBufB, xin, k == S - 1 ? kBufNone : xout, xin,
            ax_epilogue ? cf(k, 0) : 0.f, 0, 0, 0, k == 0, k == S - 1);
  }
  // Gram-space form: G = X0 X0^T; per step P = a I + b G + c G^2, Q <- P Q, G <- (P G) P; X = Q X0
  for (size_t ch = 0; ch < P.chunks.size(); ++ch) {
    if (!P.chunk_gram[ch]) continue;
    const int c = static_cast<int>(ch);
    add(DMUON_KIND_GRAM, kPhaseGram, 0, c, kListGram, kBufX0, kBufX0, kBufA, kBufNone, 0, 0, 0, 0, 1, 0);
    auto qbuf = [](int j) { return (j & 1) ? kBufQ1 : kBufQ0; };  // Q_k lives in qbuf(k + 1), k >= 1
    for (int k = 0; k < S; ++k) {
      const int pk = (k == 0) ? kBufQ0 : kBufB;
      add(DMUON_KIND_POLY, kPhasePoly, k, c, kListPoly, kBufA, kBufA, pk, kBufA, 0, cf(k, 1), cf(k, 2), cf(k, 0), 0,
          0);
      if (k >= 1) add(DMUON_KIND_SYMM, kPhaseGram, k, c, kListPoly, pk, qbuf(k + 1), qbuf(k), kBufNone, 0, 0, 0, 0, 0, 0);
      if (k < S - 1) {
        add(DMUON_KIND_SYMM, kPhaseGram, k, c, kListPoly, pk, kBufA, kBufR, kBufNone, 0, 0, 0, 0, 0, 0);
        add(DMUON_KIND_SYMM, kPhaseGram, k, c, kListPoly, kBufR, pk, kBufA, kBufNone, 0, 0, 0, 0, 0, 0);
      }
    }
    add(DMUON_KIND_GEMM, kPhaseGemm, S - 1, c, kListGemm, qbuf(S + 1), kBufX0, kBufNone, kBufX0, 0.f, 0, 0, 0, 1, 1);
  }
  // the launches that write W: the update kernel (ns_steps = 0) or the last product of each chunk
  P.first_w_launch = P.last_w_launch = -1;
  for (size_t l = 0; l < P.launches.size(); ++l) {
    const Launch& x = P.launches[l];
    if (x.kind == DMUON_KIND_UPDATE0 || (x.kind == DMUON_KIND_GEMM && x.last)) {
      if (P.first_w_launch < 0) P.first_w_launch = static_cast<int>(l);
      P.last_w_launch = static_cast<int>(l);
    }
  }
  return DMUON_OK;
}

dmuon_status make_map(CUtensorMap* map, const void* base, int inner, int rows, int count, int ld_elems,
                      int box_inner, int box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)ld_elems * 2, (cuuint64_t)ld_elems * 2 * rows};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DMUON_OK;
}

// The MN-major m x n operand of the gemm (rows of ld elements, ld a multiple of 64) as a 4-D map
// [count][chunk of 64 columns][row][64 columns], so that one box {64, 64 rows, chunks} brings a
// whole 64-row slab of chunks x 64 columns in one copy, each 64-column chunk an 8 KB block of
// 128-byte swizzled rows. Columns past n inside the last chunk read the row's padding (they feed
// only output columns past n, which are never stored); chunks past the last are zero fill.
dmuon_status make_map_mn(CUtensorMap* map, const void* base, int rows, int count, int ld_elems, int chunks_per_box) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (ld_elems % 64 != 0) return fail(DMUON_ERR_INVALID_ARG, "internal: MN-major row pitch %d not a multiple of 64", ld_elems);
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(ld_elems / 64), (cuuint64_t)count};
  cuuint64_t strides[3] = {(cuuint64_t)ld_elems * 2, 128, (cuuint64_t)ld_elems * 2 * rows};
  cuuint32_t box[4] = {64, 64, (cuuint32_t)chunks_per_box, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled failed for a 4-D operand (%d)", (int)r);
  return DMUON_OK;
}

// W (rows x cols bf16, row-major) as a 2-D map of 32 x 32 boxes with the 64-byte swizzle, for
// the TMA stores of the last step's W update. All zeros when the row pitch is not a multiple of
// 16 bytes: the kernels then update that W row by row and never use the map.
dmuon_status make_wmap(CUtensorMap* map, const void* W, int rows, int cols) {
  std::memset(map, 0, sizeof(CUtensorMap));
  if (cols % 8 != 0) return DMUON_OK;
  auto enc = get_encode_fn();
  if (enc == nullptr) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix (%d)", (int)r);
  return DMUON_OK;
}

// A bucket buffer seen as [count][rows][inner] with row pitch ld.
struct View {
  char* base;
  int inner, rows, ld;
  int64_t mat_bytes;
};

View view_of(const dmuon_plan_s& P, const BucketPlan& B, int role) {
  View v{nullptr, 0, 0, 0, 0};
  if (role == kBufNone || B.off[role] < 0) return v;
  v.base = P.ws + B.off[role];
  v.rows = B.m;
  if (B.is_x(role)) {
    v.inner = B.n;
    v.ld = B.x_ld;
    v.mat_bytes = B.x_mat_bytes;
  } else {
    v.inner = B.m;
    v.ld = B.m_ld;
    v.mat_bytes = B.a_mat_bytes;
  }
  return v;
}

// Operand maps and epilogue pointers of one bucket for one tensor-core launch.
dmuon_status fill_tc_bucket(const dmuon_plan_s& P, const BucketPlan& B, int phase, int bn, int opA, int opB,
                            int out, int aux, TcBucket& tb) {
  tb.slot_mat = reinterpret_cast<const int32_t*>(P.ws + B.off_slotmat);
  tb.m = B.m;
  tb.n = B.n;
  const View va = view_of(P, B, opA), vb = view_of(P, B, opB), vo = view_of(P, B, out), vx = view_of(P, B, aux);
  dmuon_status st = make_map(&tb.tmA, va.base, va.inner, va.rows, B.count, va.ld, 64, kTcBM);
  if (st != DMUON_OK) return st;
  if (phase == kPhaseGemm)  // the m x n operand, MN-major: bn/64 chunks of 64 columns x 64 rows per box
    st = make_map_mn(&tb.tmB, vb.base, vb.rows, B.count, vb.ld, bn / 64);
  else
    st = make_map(&tb.tmB, vb.base, vb.inner, vb.rows, B.count, vb.ld, 64, bn);
  if (st != DMUON_OK) return st;
  tb.kdim = (phase == kPhaseGemm) ? B.m : va.inner;
  tb.same_ab = (phase != kPhaseGemm && opA == opB) ? 1 : 0;
  if (vo.base != nullptr) {  // epilogue stores: 32 x 32 boxes staged with a 64-byte swizzle
    st = make_map(&tb.tmOut, vo.base, vo.inner, vo.rows, B.count, vo.ld, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != DMUON_OK) return st;
  }
  tb.out = vo.base;
  tb.out_mat_stride = vo.mat_bytes;
  tb.out_ld = vo.ld;
  tb.aux = vx.base;
  tb.aux_mat_stride = vx.mat_bytes;
  tb.aux_ld = vx.ld;
  return DMUON_OK;
}

dmuon_status record_launch(dmuon_plan_s& P, const Launch& L, cudaStream_t s, bool before) {
  if (!P.prof || P.prof_n >= P.prof_max) return DMUON_OK;
  cudaError_t e;
  if (before) {
    e = cudaEventRecord(P.ev_start[P.prof_n], s);
  } else {
    e = cudaEventRecord(P.ev_stop[P.prof_n], s);
    P.prof_kind[P.prof_n] = L.kind;
    P.prof_work[P.prof_n] = L.work;
    ++P.prof_n;
  }
  return e == cudaSuccess ? DMUON_OK : cuda_fail(e, "cudaEventRecord");
}

void destroy_events(dmuon_plan_s& P) {
  for (auto e : P.ev_start) cudaEventDestroy(e);
  for (auto e : P.ev_stop) cudaEventDestroy(e);
  P.ev_start.clear();
  P.ev_stop.clear();
  P.prof = false;
  P.prof_max = P.prof_n = 0;
}

// Init-time tuning (DMUON_FLAG_TUNE): for every bucket and every tile
// configuration (one-SM 128 x 128 tiles with a 6-stage ring, one-SM 128 x 256
// with 4 stages, and, where the short side is at least 256, two-SM 256 x 256
// pairs with 6 stages), time a GPU-filling slice of its X X^T tiles (K = n),
// of its m x m products (K = m) and of its gemm tiles on the bound workspace
// (results discarded), keep the cheapest configuration per bucket, and record
// the measured SM-time per tile, which then orders the tile lists and feeds
// dmuon_plan_costs. The per-tile times are kept in a process-wide cache keyed
// by (short side, long side, weight dtype, SM count, compute capability), so
// later plans with the same shapes bind without timing again. This is the
// single-GPU form of the pages' initialisation profiling of kernel schedules
// per matrix shape ("DMuon: Efficient Distributed Muon Training with
// Near-Adam Overhead", gist.science summary section 2.3, "Profiling";
// section 2.4: tile shapes, block sizes and pipeline depths are searched and
// the chosen configuration is cached and reused).
constexpr int kTuneCands = 3;  // 0: one-SM 128 wide, 1: one-SM 256 wide, 2: two-SM 256 x 256
constexpr double kTuneHeatMs = 150.0, kTuneTimedMs = 150.0;  // per configuration and kind of product
constexpr double kTuneMargin = 0.05;  // a configuration other than the default must be this much cheaper
constexpr int kTuneCandBn[kTuneCands] = {128, 256, 256};

struct TuneKey {
  int m, n, param, sms, cc;
  bool operator<(const TuneKey& o) const {
    return std::tie(m, n, param, sms, cc) < std::tie(o.m, o.n, o.param, o.sms, o.cc);
  }
};
struct TuneTimes {
  double sm_ms[kTuneCands][3];  // SM-ms per tile: X X^T, m x m product, gemm; 0 = candidate not timed
};
std::mutex g_tune_mu;
std::map<TuneKey, TuneTimes> g_tune_cache;

dmuon_status tune_plan(dmuon_plan_s& P, cudaStream_t s) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e;
  if ((e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    return cuda_fail(e, "cudaEventCreate");
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, P.device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, P.device);
  dmuon_status st = DMUON_OK;
  int4* probe = reinterpret_cast<int4*>(P.ws + P.off_probe);
  std::vector<int4> tiles;
  P.tune_timed = P.tune_cached = 0;
  for (BucketPlan& B : P.buckets) {
    const TuneKey key{B.m, B.n, P.dt.param, P.num_sms, 10 * major + minor};
    TuneTimes tt{};
    bool cached = false;
    {
      std::lock_guard<std::mutex> lock(g_tune_mu);
      auto it = g_tune_cache.find(key);
      if (it != g_tune_cache.end()) {
        tt = it->second;
        cached = true;
      }
    }
    if (!cached) {
      // realistic operands for the probes: X0 and A of the first slots the probes touch
      const int slots = std::min(B.count, 8);
      if ((e = launch_tuning_fill(P.ws + B.off[kBufX0], B.x_mat_bytes * slots, 17u, 4 * P.num_sms, s)) !=
              cudaSuccess ||
          (e = launch_tuning_fill(P.ws + B.off[kBufA], B.a_mat_bytes * slots, 29u, 4 * P.num_sms, s)) != cudaSuccess) {
        st = cuda_fail(e, "tuning fill");
        break;
      }
    }
    for (int ci = 0; ci < kTuneCands && st == DMUON_OK && !cached; ++ci) {
      BucketPlan T = B;
      T.bn_sym = T.bn_gemm = kTuneCandBn[ci];
      T.pair = (ci == 2);
      if (T.pair && B.m < 256) continue;  // a pair tile would be mostly empty
      for (int kind = 0; kind < 3 && st == DMUON_OK; ++kind) {
        tiles.clear();
        add_tiles(P, kind == 2 ? DMUON_KIND_GEMM : DMUON_KIND_GRAM, 0, T, tiles);
        const int slots = T.pair ? P.num_sms / 2 : P.num_sms;
        const int n = static_cast<int>(std::min<int64_t>({(int64_t)tiles.size(), 4LL * slots, kProbeTiles}));
        if ((e = cudaMemcpyAsync(probe, tiles.data(), sizeof(int4) * n, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
            (e = cudaStreamSynchronize(s)) != cudaSuccess) {
          st = cuda_fail(e, "probe upload");
          break;
        }
        int phase, opA, opB, out, aux = kBufNone;
        if (kind == 0) {
          phase = kPhaseGram, opA = opB = kBufX0, out = kBufA;
        } else if (kind == 1) {
          phase = kPhaseGram, opA = opB = kBufA, out = B.off[kBufB] >= 0 ? kBufB : kBufQ0;
        } else {  // the output goes to a buffer that no probe reads (values unused, only the time)
          const int spare = B.off[kBufX1] >= 0 ? kBufX1 : (B.off[kBufR] >= 0 ? kBufR : kBufX0);
          phase = kPhaseGemm, opA = kBufA, opB = kBufX0, out = spare, aux = kBufX0;
        }
        TcParams tp;
        std::memset(&tp, 0, sizeof(tp));
        // a pair's CTAs each load 128 rows of a K-major B operand
        if ((st = fill_tc_bucket(P, T, phase, T.pair ? 128 : T.bn_sym, opA, opB, out, aux, tp.bk[0])) != DMUON_OK)
          break;
        tp.items = probe;
        tp.n_items = n;
        tp.a = 1.f;
        tp.mats = P.sp.mats;
        tp.ptrs = P.sp.ptrs;
        tp.s_norm = P.sp.s_norm;
        tp.status = P.sp.status;
        tp.param_bf16 = P.sp.param_bf16;
        tp.timeout_ns = 2000000000LL;
        tp.sched = (P.flags & DMUON_FLAG_STATIC_TILES) ? nullptr
                                                        : reinterpret_cast<unsigned*>(P.ws + P.off_probe_sched);
        const int grid = std::max(1, std::min(n, slots));
        auto launch = [&]() {
          return T.pair ? launch_tc_pair(phase, tp, grid, s) : launch_tc(phase, T.bn_sym, tp, grid, s);
        };
        // Timed long enough for the clock to settle under the power limit: about 150 ms untimed,
        // then about 150 ms timed. A configuration that does more work per clock but draws more
        // power is then measured closer to the clock it gets in a long step than to an idle GPU's.
        auto run = [&](int reps, float* ms) -> cudaError_t {
          cudaError_t r = cudaEventRecord(e0, s);
          for (int rep = 0; rep < reps && r == cudaSuccess; ++rep) r = launch();
          if (r == cudaSuccess) r = cudaEventRecord(e1, s);
          if (r == cudaSuccess) r = cudaEventSynchronize(e1);
          if (r == cudaSuccess) r = cudaEventElapsedTime(ms, e0, e1);
          return r;
        };
        float ms = 0.f;
        e = run(1, &ms);  // also the first launch of this kernel
        const double per = std::max(ms, 0.01f);
        if (e == cudaSuccess) e = run(static_cast<int>(std::min(2000.0, std::ceil(kTuneHeatMs / per))), &ms);
        const int reps = static_cast<int>(std::min(2000.0, std::max(3.0, std::ceil(kTuneTimedMs / per))));
        if (e == cudaSuccess) e = run(reps, &ms);
        if (e != cudaSuccess) {
          st = cuda_fail(e, "tuning run");
          break;
        }
        const int waves = (n + grid - 1) / grid;
        tt.sm_ms[ci][kind] = ms / reps / waves * (T.pair ? 2.0 : 1.0);  // SMs a tile occupies
      }
    }
    if (st != DMUON_OK) break;
    if (cached) {
      ++P.tune_cached;
    } else {
      ++P.tune_timed;
      std::lock_guard<std::mutex> lock(g_tune_mu);
      g_tune_cache[key] = tt;
    }
    // cost per matrix of each configuration: tiles x SM-ms per tile, for the products this bucket's
    // form runs (the Gram-space form: one X X^T, 4S - 3 m x m products, one gemm)
    const double S = P.ns_steps;
    const double n_xx = B.gram ? 1.0 : S, n_mm = B.gram ? 4.0 * S - 3.0 : S, n_gm = B.gram ? 1.0 : S;
    double cs[kTuneCands], cg[kTuneCands];
    for (int ci = 0; ci < kTuneCands; ++ci) {
      BucketPlan T = B;
      T.bn_sym = T.bn_gemm = kTuneCandBn[ci];
      T.pair = (ci == 2);
      T.count = 1;
      cs[ci] = cg[ci] = 1e300;
      if (tt.sm_ms[ci][0] <= 0 || tt.sm_ms[ci][1] <= 0 || tt.sm_ms[ci][2] <= 0) continue;
      tiles.clear();
      add_tiles(P, DMUON_KIND_GRAM, 0, T, tiles);
      cs[ci] = tiles.size() * (n_xx * tt.sm_ms[ci][0] + n_mm * tt.sm_ms[ci][1]);
      tiles.clear();
      add_tiles(P, DMUON_KIND_GEMM, 0, T, tiles);
      cg[ci] = tiles.size() * n_gm * tt.sm_ms[ci][2];
    }
    for (int ci = 0; ci < kTuneCands; ++ci) {
      B.tune_cost[ci] = cs[ci] + cg[ci] < 1e299 ? cs[ci] + cg[ci] : 0.0;
      B.tune_gemm[ci] = cg[ci] < 1e299 ? cg[ci] : 0.0;
    }
    // Best one-SM widths, then pairs against them. A configuration other than the planner's default
    // must be cheaper by kTuneMargin: what a probe gains per clock, a long step under the power limit
    // partly gives back in clock (measured: pairs chosen on a 2 % probe advantage lost 5 % on MoE).
    const int dsym = B.bn_sym == 128 ? 0 : 1, dgem = B.bn_gemm == 128 ? 0 : 1;  // the default widths
    const int bs = cs[1 - dsym] * (1.0 + kTuneMargin) < cs[dsym] ? 1 - dsym : dsym;
    const int bg = cg[1 - dgem] * (1.0 + kTuneMargin) < cg[dgem] ? 1 - dgem : dgem;
    const double best_one = cs[bs] + cg[bg], dflt = cs[dsym] + cg[dgem];
    const bool dflt_pair = B.pair;
    const double pair_cost = cs[2] + cg[2];
    if (dflt_pair ? !(best_one * (1.0 + kTuneMargin) < pair_cost)
                  : (pair_cost * (1.0 + kTuneMargin) < dflt && pair_cost < best_one)) {
      B.pair = true;
      B.bn_sym = B.bn_gemm = 256;
      for (int k = 0; k < 3; ++k) B.tile_ms[k] = tt.sm_ms[2][k];
    } else {
      B.pair = false;
      B.bn_sym = kTuneCandBn[bs];
      B.bn_gemm = kTuneCandBn[bg];
      B.tile_ms[0] = tt.sm_ms[bs][0];
      B.tile_ms[1] = tt.sm_ms[bs][1];
      B.tile_ms[2] = tt.sm_ms[bg][2];
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != DMUON_OK) return st;
  P.tuned = true;
  // re-plan with the chosen configurations; the workspace layout the caller sized must not move
  std::vector<int64_t> before;
  for (const BucketPlan& B : P.buckets) before.insert(before.end(), std::begin(B.off), std::end(B.off));
  before.insert(before.end(), {P.off_items, P.off_sched, P.off_cta, P.off_capture, (int64_t)P.ws_bytes});
  if ((st = finish_plan(P)) != DMUON_OK) return st;
  std::vector<int64_t> after;
  for (const BucketPlan& B : P.buckets) after.insert(after.end(), std::begin(B.off), std::end(B.off));
  after.insert(after.end(), {P.off_items, P.off_sched, P.off_cta, P.off_capture, (int64_t)P.ws_bytes});
  if (after != before) return fail(DMUON_ERR_WORKSPACE, "internal: tuning moved the workspace layout");
  return DMUON_OK;
}

// ------------------------------------------------------------------ debug checks
// DMUON_FLAG_DEBUG_CHECKS: after every launch of a step the host waits for it,
// copies back the operands of a few sampled output elements and recomputes
// them in double precision; the step fails with DMUON_ERR_DEVICE and a message
// naming the launch, the matrix and the element when one is off by more than
// the rounding of the stored result allows. Sampled per launch: the momentum
// and U of two elements of three matrices; s of the smallest matrix; for each
// product two random elements, one diagonal element and, for the symmetric
// products, the mirror of a random element (which must be bit-identical); for
// the last product, the updated weights of its samples.

struct DbgRng {
  uint64_t s;
  uint32_t next() {
    s = s * 6364136223846793005ULL + 1442695040888963407ULL;
    return static_cast<uint32_t>(s >> 33);
  }
  int below(int n) { return n > 0 ? static_cast<int>(next() % static_cast<uint32_t>(n)) : 0; }
};

double decode(const unsigned char* p, int el) {
  if (el == 2) {
    uint16_t h;
    std::memcpy(&h, p, 2);
    const uint32_t w = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &w, 4);
    return f;
  }
  float f;
  std::memcpy(&f, p, 4);
  return f;
}

// count elements of `el` bytes starting at dptr, stride_el elements apart, into out (as doubles).
dmuon_status dbg_read(const char* dptr, int64_t count, int el, int64_t stride_el, std::vector<double>& out,
                      cudaStream_t s) {
  std::vector<unsigned char> h(static_cast<size_t>(count) * el);
  cudaError_t e = stride_el == 1
                      ? cudaMemcpyAsync(h.data(), dptr, h.size(), cudaMemcpyDeviceToHost, s)
                      : cudaMemcpy2DAsync(h.data(), el, dptr, static_cast<size_t>(stride_el) * el, el, count,
                                          cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "debug-check copy");
  out.resize(count);
  for (int64_t k = 0; k < count; ++k) out[k] = decode(h.data() + k * el, el);
  return DMUON_OK;
}

double dbg_one(const char* dptr, int el, cudaStream_t s, dmuon_status& st) {
  std::vector<double> v;
  st = dbg_read(dptr, 1, el, 1, v, s);
  return st == DMUON_OK ? v[0] : 0.0;
}

// True when got differs from want by more than tol, or is not finite while want is (a non-finite
// want cannot be checked: it comes from non-finite inputs, which the kernels propagate).
bool off_by(double got, double want, double tol) {
  return std::isfinite(want) && !(std::fabs(got - want) <= tol);
}

struct DbgSample {
  int bucket = 0, slot = 0, gm = 0, i = 0, j = 0;
  int64_t w_off = 0;  // element offset of W(i, j) or of the sampled element (momentum pass)
  double pre_w = 0, pre_g = 0, pre_m = 0;
  bool mirror = false;  // symmetric products: (i, j) is checked against its mirror (j, i)
};

double ulp_of(double x, int el) {
  const int bits = el == 2 ? 8 : 24;
  const double ax = std::max(std::fabs(x), 1e-38);
  return std::ldexp(1.0, static_cast<int>(std::floor(std::log2(ax))) - (bits - 1));
}

dmuon_status dbg_mismatch(const dmuon_plan_s& P, int li, const Launch& L, const DbgSample& x, const char* what,
                          double got, double want, double tol) {
  return fail(DMUON_ERR_DEVICE,
              "debug check: launch %d (kind %d, step %d) matrix %d (%d x %d) %s at (%d, %d): got %.9g, expected "
              "%.9g (tolerance %.3g)",
              li, L.kind, L.step, x.gm, P.mats[x.gm].rows, P.mats[x.gm].cols, what, x.i, x.j, got, want, tol);
}

dmuon_status debug_before(dmuon_plan_s& P, const Launch& L, int li, void* const* params, const void* const* grads,
                          void* const* momenta, std::vector<DbgSample>& smp, cudaStream_t s) {
  smp.clear();
  DbgRng rng{0x9E3779B97F4A7C15ULL ^ (static_cast<uint64_t>(P.steps_taken) << 20) ^ static_cast<uint64_t>(li)};
  dmuon_status st = DMUON_OK;
  const int gb = dtype_bytes(P.dt.grad), pb = dtype_bytes(P.dt.param);
  if (L.kind == DMUON_KIND_MOMENTUM) {
    const int n = static_cast<int>(P.mats.size());
    const int picks[3] = {0, n - 1, rng.below(n)};
    for (int gm : picks)
      for (int e = 0; e < 2; ++e) {
        DbgSample x;
        x.gm = gm;
        x.i = rng.below(P.mats[gm].rows);
        x.j = rng.below(P.mats[gm].cols);
        x.w_off = static_cast<int64_t>(x.i) * P.mats[gm].cols + x.j;
        x.pre_g = dbg_one(static_cast<const char*>(grads[gm]) + x.w_off * gb, gb, s, st);
        if (st == DMUON_OK) x.pre_m = dbg_one(static_cast<const char*>(momenta[gm]) + x.w_off * 4, 4, s, st);
        if (st != DMUON_OK) return st;
        smp.push_back(x);
      }
    return DMUON_OK;
  }
  if (L.kind == DMUON_KIND_NORM || L.kind == DMUON_KIND_UPDATE0) {
    // the smallest matrix: its s (norm) or every weight of one row (update)
    int best = 0;
    for (size_t k = 1; k < P.mats.size(); ++k)
      if ((int64_t)P.mats[k].rows * P.mats[k].cols < (int64_t)P.mats[best].rows * P.mats[best].cols) best = (int)k;
    DbgSample x;
    x.gm = best;
    x.i = rng.below(P.mats[best].rows);
    x.j = rng.below(P.mats[best].cols);
    x.w_off = static_cast<int64_t>(x.i) * P.mats[best].cols + x.j;
    if (L.kind == DMUON_KIND_UPDATE0) x.pre_w = dbg_one(static_cast<const char*>(params[best]) + x.w_off * pb, pb, s, st);
    smp.push_back(x);
    return st;
  }
  const std::vector<int>& ch = P.chunks[L.chunk];
  const bool sym = L.phase != kPhaseGemm;
  for (int q = 0; q < 4; ++q) {
    DbgSample x;
    const int lb = rng.below(static_cast<int>(ch.size()));
    const BucketPlan& B = P.buckets[ch[lb]];
    x.bucket = lb;
    x.slot = rng.below(B.count);
    x.gm = B.mats[x.slot];
    const int ncols = sym ? B.m : B.n;
    x.i = rng.below(B.m);
    x.j = (q == 2) ? std::min(x.i, ncols - 1) : rng.below(ncols);
    x.mirror = sym && q == 3 && x.i != x.j;
    if (L.last) {
      const MatDev& md = P.mats[x.gm];
      x.w_off = md.transposed ? static_cast<int64_t>(x.j) * md.cols + x.i : static_cast<int64_t>(x.i) * md.cols + x.j;
      x.pre_w = dbg_one(static_cast<const char*>(params[x.gm]) + x.w_off * pb, pb, s, st);
      if (st != DMUON_OK) return st;
    }
    smp.push_back(x);
  }
  return DMUON_OK;
}

dmuon_status debug_after(dmuon_plan_s& P, const Launch& L, int li, void* const* params, void* const* momenta,
                         const std::vector<DbgSample>& smp, float lr, float mu, int nesterov, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "debug-check sync");
  dmuon_status st = DMUON_OK;
  const int el = P.xel, pb = dtype_bytes(P.dt.param);
  const double f32 = std::ldexp(1.0, -22);
  auto s_of = [&](int gm) { return dbg_one(P.ws + P.off_s + 4LL * gm, 4, s, st); };
  if (L.kind == DMUON_KIND_MOMENTUM) {
    for (const DbgSample& x : smp) {
      const MatDev& md = P.mats[x.gm];
      const double m_got = dbg_one(static_cast<const char*>(momenta[x.gm]) + x.w_off * 4, 4, s, st);
      const int64_t u_off = md.transposed ? static_cast<int64_t>(x.j) * md.x_ld + x.i
                                          : static_cast<int64_t>(x.i) * md.x_ld + x.j;
      const double u_got = st == DMUON_OK ? dbg_one(P.ws + md.x0_off + u_off * el, el, s, st) : 0.0;
      if (st != DMUON_OK) return st;
      const double m_want = mu * x.pre_m + x.pre_g;
      const double tm = f32 * (std::fabs(mu * x.pre_m) + std::fabs(x.pre_g)) + 1e-38;
      if (off_by(m_got, m_want, tm)) return dbg_mismatch(P, li, L, x, "momentum", m_got, m_want, tm);
      const double u_want = nesterov ? x.pre_g + mu * m_got : m_got;
      const double tu = (el == 2 ? ulp_of(u_want, 2) : 0.0) + f32 * (std::fabs(x.pre_g) + std::fabs(mu * m_got)) + 1e-38;
      if (off_by(u_got, u_want, tu)) return dbg_mismatch(P, li, L, x, "U", u_got, u_want, tu);
    }
    return DMUON_OK;
  }
  if (L.kind == DMUON_KIND_NORM) {
    const DbgSample& x = smp[0];
    const MatDev& md = P.mats[x.gm];
    std::vector<double> row;
    double ss = 0;
    for (int r = 0; r < md.m && st == DMUON_OK; ++r) {
      st = dbg_read(P.ws + md.x0_off + static_cast<int64_t>(r) * md.x_ld * el, md.n, el, 1, row, s);
      for (double v : row) ss += v * v;
    }
    const double got = s_of(x.gm);
    if (st != DMUON_OK) return st;
    const double want = 1.0 / (std::sqrt(ss) + P.eps);
    const double tol = (el == 2 ? std::ldexp(1.0, -7) : 1e-5) * want;
    if (off_by(got, want, tol)) return dbg_mismatch(P, li, L, x, "s = 1/(|U|+eps)", got, want, tol);
    return DMUON_OK;
  }
  if (L.kind == DMUON_KIND_UPDATE0) {
    const DbgSample& x = smp[0];
    const MatDev& md = P.mats[x.gm];
    const int64_t u_off = md.transposed ? static_cast<int64_t>(x.j) * md.x_ld + x.i : static_cast<int64_t>(x.i) * md.x_ld + x.j;
    const double u = dbg_one(P.ws + md.x0_off + u_off * el, el, s, st);
    const double sn = st == DMUON_OK ? s_of(x.gm) : 0.0;
    const double got = st == DMUON_OK ? dbg_one(static_cast<const char*>(params[x.gm]) + x.w_off * pb, pb, s, st) : 0.0;
    if (st != DMUON_OK) return st;
    const double want = x.pre_w - static_cast<double>(lr) * md.scale * sn * u;
    const double tol = ulp_of(want, pb) + f32 * (std::fabs(x.pre_w) + std::fabs(lr * md.scale * sn * u)) + 1e-38;
    if (off_by(got, want, tol)) return dbg_mismatch(P, li, L, x, "updated weight", got, want, tol);
    return DMUON_OK;
  }
  const std::vector<int>& ch = P.chunks[L.chunk];
  std::vector<double> ra, rb;
  for (const DbgSample& x : smp) {
    const BucketPlan& B = P.buckets[ch[x.bucket]];
    const MatDev& md = P.mats[x.gm];
    const View va = view_of(P, B, L.opA), vb = view_of(P, B, L.opB), vx = view_of(P, B, L.aux);
    const int K = L.phase == kPhaseGemm ? B.m : va.inner;
    // row i of the first operand; row j (symmetric products) or column j (gemm) of the second. A
    // symmetric product is computed on the upper element (r, c), r <= c, and mirrored, so the
    // element at (i, j) is the one computed from rows min(i, j) and max(i, j): with two different
    // operands (the Gram-space form) the two orders differ by the operands' rounding.
    const bool sym = L.phase != kPhaseGemm;
    const int r = sym ? std::min(x.i, x.j) : x.i, c = sym ? std::max(x.i, x.j) : x.j;
    st = dbg_read(va.base + x.slot * va.mat_bytes + static_cast<int64_t>(r) * va.ld * el, K, el, 1, ra, s);
    if (st == DMUON_OK) {
      if (L.phase == kPhaseGemm)
        st = dbg_read(vb.base + x.slot * vb.mat_bytes + static_cast<int64_t>(c) * el, K, el, vb.ld, rb, s);
      else
        st = dbg_read(vb.base + x.slot * vb.mat_bytes + static_cast<int64_t>(c) * vb.ld * el, K, el, 1, rb, s);
    }
    if (st != DMUON_OK) return st;
    double acc = 0, mag = 0;
    for (int k = 0; k < K; ++k) {
      acc += ra[k] * rb[k];
      mag += std::fabs(ra[k] * rb[k]);
    }
    const double sn = L.first ? s_of(x.gm) : 1.0;
    if (st != DMUON_OK) return st;
    double want, tol;
    const double acc_err = std::ldexp(1.0, -20) * mag;  // fp32 accumulation over K, generously
    if (L.kind == DMUON_KIND_POLY) {
      const double a = dbg_one(vx.base + x.slot * vx.mat_bytes + (static_cast<int64_t>(x.i) * vx.ld + x.j) * el, el, s, st);
      want = L.b * a + L.c * acc + (x.i == x.j ? L.diag : 0.0);
      tol = std::fabs(L.c) * acc_err + f32 * (std::fabs(L.b * a) + std::fabs(L.c * acc) + std::fabs(L.diag));
    } else if (L.phase != kPhaseGemm) {  // X X^T (scaled by s^2 at step 0) or a product of two symmetric matrices
      want = (L.kind == DMUON_KIND_GRAM && L.first ? sn * sn : 1.0) * acc;
      tol = (L.kind == DMUON_KIND_GRAM && L.first ? sn * sn : 1.0) * acc_err;
    } else {
      double ax = 0;
      if (L.a != 0.f)
        ax = dbg_one(vx.base + x.slot * vx.mat_bytes + (static_cast<int64_t>(x.i) * vx.ld + x.j) * el, el, s, st);
      want = sn * (acc + L.a * ax);
      tol = sn * (acc_err + f32 * (std::fabs(acc) + std::fabs(L.a * ax)));
    }
    if (st != DMUON_OK) return st;
    if (!L.last) {
      const View vo = view_of(P, B, L.out);
      const char* po = vo.base + x.slot * vo.mat_bytes;
      const double got = dbg_one(po + (static_cast<int64_t>(x.i) * vo.ld + x.j) * el, el, s, st);
      if (st != DMUON_OK) return st;
      const double t = tol + ulp_of(want, el) + 1e-38;
      if (off_by(got, want, t)) return dbg_mismatch(P, li, L, x, "product", got, want, t);
      if (x.mirror) {  // the mirrored element holds the same stored value, bit for bit
        const double mir = dbg_one(po + (static_cast<int64_t>(x.j) * vo.ld + x.i) * el, el, s, st);
        if (st != DMUON_OK) return st;
        if (!(mir == got)) return dbg_mismatch(P, li, L, x, "mirror (j, i) of the product", mir, got, 0.0);
      }
    } else {  // the weight update of the last product
      const double step = static_cast<double>(lr) * md.scale;
      const double got = dbg_one(static_cast<const char*>(params[x.gm]) + x.w_off * pb, pb, s, st);
      if (st != DMUON_OK) return st;
      const double wwant = x.pre_w - step * want;
      const double t = ulp_of(wwant, pb) + step * tol + f32 * (std::fabs(x.pre_w) + std::fabs(step * want)) + 1e-38;
      if (off_by(got, wwant, t)) return dbg_mismatch(P, li, L, x, "updated weight", got, wwant, t);
    }
  }
  return DMUON_OK;
}

}  // namespace

dmuon_status dmuon::set_last_error(dmuon_status st, const char* msg) {
  g_err = msg;
  return st;
}

// ============================================================================ C ABI
extern "C" {

int32_t dmuon_version(void) { return 100; }

const char* dmuon_last_error(void) { return g_err.c_str(); }

dmuon_status dmuon_plan(const dmuon_shape* shapes, int32_t n_mats, int32_t ns_steps, const float* coeffs,
                        int32_t n_coeff_triples, float eps, dmuon_dtypes dtypes, uint32_t flags,
                        dmuon_plan_t* out) {
  g_err.clear();
  if (out == nullptr) return fail(DMUON_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (shapes == nullptr || n_mats <= 0) return fail(DMUON_ERR_INVALID_ARG, "empty matrix list");
  if (ns_steps < 0 || ns_steps > 16) return fail(DMUON_ERR_INVALID_ARG, "ns_steps %d outside 0..16", ns_steps);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(DMUON_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (flags & ~(DMUON_FLAG_CAPTURE_UPDATE | DMUON_FLAG_GRAM_NS | DMUON_FLAG_TUNE | DMUON_FLAG_PAIR_TILES |
                DMUON_FLAG_EPILOGUE_AX | DMUON_FLAG_STATIC_TILES | DMUON_FLAG_DEBUG_CHECKS | DMUON_FLAG_ONE_SM_TILES))
    return fail(DMUON_ERR_UNSUPPORTED, "unknown flag bits 0x%x", flags);
  if ((flags & DMUON_FLAG_ONE_SM_TILES) && (flags & (DMUON_FLAG_PAIR_TILES | DMUON_FLAG_TUNE)))
    return fail(DMUON_ERR_INVALID_ARG, "DMUON_FLAG_ONE_SM_TILES excludes DMUON_FLAG_PAIR_TILES and DMUON_FLAG_TUNE");
  for (int32_t d : {dtypes.param, dtypes.grad, dtypes.compute})
    if (d != DMUON_F32 && d != DMUON_BF16) return fail(DMUON_ERR_UNSUPPORTED, "unknown dtype %d", d);
  if (dtypes.momentum != DMUON_F32) return fail(DMUON_ERR_UNSUPPORTED, "momentum must be DMUON_F32");
  for (int32_t i = 0; i < n_mats; ++i) {
    const int64_t r = shapes[i].rows, c = shapes[i].cols;
    if (r < 1 || c < 1 || r > (1 << 20) || c > (1 << 20) || r * c >= (1LL << 31))
      return fail(DMUON_ERR_INVALID_ARG, "matrix %d has unsupported shape %lld x %lld", i, (long long)r,
                  (long long)c);
  }
  std::vector<float> cf;
  if (n_coeff_triples == 0 && coeffs == nullptr) {
    for (int k = 0; k < ns_steps; ++k) cf.insert(cf.end(), {3.4445f, -4.7750f, 2.0315f});
  } else {
    if (coeffs == nullptr) return fail(DMUON_ERR_INVALID_ARG, "coeffs is NULL");
    if (n_coeff_triples != 1 && n_coeff_triples != ns_steps)
      return fail(DMUON_ERR_INVALID_ARG, "n_coeff_triples must be 1 or ns_steps");
    for (int k = 0; k < ns_steps; ++k) {
      const float* t = coeffs + 3 * (n_coeff_triples == 1 ? 0 : k);
      for (int q = 0; q < 3; ++q)
        if (!std::isfinite(t[q])) return fail(DMUON_ERR_INVALID_ARG, "non-finite coefficient");
      cf.insert(cf.end(), {t[0], t[1], t[2]});
    }
  }
  auto* P = new (std::nothrow) dmuon_plan_s();
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "out of host memory");
  P->shapes.assign(shapes, shapes + n_mats);
  P->ns_steps = ns_steps;
  P->coeffs = cf;
  P->eps = eps;
  P->dt = dtypes;
  P->flags = flags;
  dmuon_status st = build_plan(*P);
  if (st != DMUON_OK) {
    delete P;
    return st;
  }
  logf("plan %p: %d matrices, %zu buckets, %zu launch chunks, %zu launches per step, ns_steps %d, compute %s, "
       "flags 0x%x, workspace %zu bytes",
       (void*)P, n_mats, P->buckets.size(), P->chunks.size(), P->launches.size(), ns_steps, P->tc ? "bf16" : "f32",
       flags, P->ws_bytes);
  for (const BucketPlan& B : P->buckets)
    logf("  bucket %d x %d: %d matrices (%d transposed), form %s, tile widths %d/%d%s", B.m, B.n, B.count,
         B.n_transposed, B.gram ? "gram" : "standard", B.bn_sym, B.bn_gemm, B.pair ? ", pairs" : "");
  *out = P;
  return DMUON_OK;
}

dmuon_status dmuon_plan_workspace_bytes(dmuon_plan_t P, size_t* bytes) {
  if (P == nullptr || bytes == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  *bytes = P->ws_bytes;
  return DMUON_OK;
}

dmuon_status dmuon_plan_bind(dmuon_plan_t P, void* d_workspace, size_t bytes, void* stream) {
  g_err.clear();
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "plan is NULL");
  // Every failing return below leaves the plan unbound (a step then returns DMUON_ERR_NOT_BOUND),
  // whether it was bound before or not: never bound to half-written tables, nor to a workspace
  // of one device with the device and SM count of another.
  struct Unbind {
    dmuon_plan_s* plan;
    bool done = false;
    ~Unbind() {
      if (!done) {
        plan->ws = nullptr;
        plan->device = -1;
      }
    }
  } unbind{P};
  if (d_workspace == nullptr) return fail(DMUON_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(d_workspace) % kAlign != 0)
    return fail(DMUON_ERR_WORKSPACE, "workspace must be %lld-byte aligned", (long long)kAlign);
  if (bytes < P->ws_bytes)
    return fail(DMUON_ERR_WORKSPACE, "workspace has %zu bytes, plan needs %zu", bytes, P->ws_bytes);
  if (test_hook("bind_check")) return fail(DMUON_ERR_CUDA, "injected failure (DMUON_TEST_FAIL=bind_check)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  int device = -1, num_sms = 0;
  if ((e = cudaGetDevice(&device)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, d_workspace) != cudaSuccess || pa.type != cudaMemoryTypeDevice ||
      pa.device != device) {
    cudaGetLastError();
    return fail(DMUON_ERR_WORKSPACE, "workspace is not device memory of the current device %d", device);
  }
  if (P->tc) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (major != 10 || minor != 3)
      return fail(DMUON_ERR_UNSUPPORTED, "bf16 compute needs an sm_103 GPU (found sm_%d%d)", major, minor);
  }
  P->ws = static_cast<char*>(d_workspace);
  P->device = device;
  P->num_sms = num_sms;
  char* ws = P->ws;

  // tables
  auto up = [&](int64_t off, const void* src, size_t n) -> cudaError_t {
    if (n == 0) return cudaSuccess;
    return cudaMemcpyAsync(ws + off, src, n, cudaMemcpyHostToDevice, s);
  };
  if ((e = up(P->off_mats, P->mats.data(), sizeof(MatDev) * P->mats.size())) != cudaSuccess ||
      (e = up(P->off_ub, P->unit_begin.data(), 8 * P->unit_begin.size())) != cudaSuccess ||
      (e = up(P->off_items, P->items.data(), sizeof(int4) * P->items.size())) != cudaSuccess)
    return cuda_fail(e, "table upload");
  for (const BucketPlan& B : P->buckets)
    if ((e = up(B.off_slotmat, B.mats.data(), 4 * B.mats.size())) != cudaSuccess) return cuda_fail(e, "upload");
  if ((e = cudaMemsetAsync(ws + P->off_status, 0, P->off_s - P->off_status, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(ws + P->off_sched, 0, P->off_cta - P->off_sched, s)) != cudaSuccess)
    return cuda_fail(e, "cudaMemsetAsync");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "bind sync");
  if (test_hook("bind_tables")) return fail(DMUON_ERR_CUDA, "injected failure (DMUON_TEST_FAIL=bind_tables)");

  // momentum-pass parameters
  StreamParams& sp = P->sp;
  sp = StreamParams{};
  sp.mats = reinterpret_cast<const MatDev*>(ws + P->off_mats);
  sp.unit_begin = reinterpret_cast<const int64_t*>(ws + P->off_ub);
  sp.ptrs = reinterpret_cast<const uint64_t*>(ws + P->off_ptrs);
  sp.ws = ws;
  sp.partial = reinterpret_cast<float*>(ws + P->off_partial);
  sp.s_norm = reinterpret_cast<float*>(ws + P->off_s);
  sp.status = reinterpret_cast<unsigned*>(ws + P->off_status);
  sp.capture = P->off_capture >= 0 ? reinterpret_cast<float*>(ws + P->off_capture) : nullptr;
  sp.n_units = P->n_units;
  sp.n_mats = static_cast<int32_t>(P->mats.size());
  sp.eps = P->eps;
  sp.grad_bf16 = P->dt.grad == DMUON_BF16;
  sp.x_bf16 = P->tc;
  sp.param_bf16 = P->dt.param == DMUON_BF16;

  // init-time tuning of tile widths and per-tile costs (needs the tables and sp above)
  if ((P->flags & DMUON_FLAG_TUNE) && P->tc && P->ns_steps > 0) {
    dmuon_status st = tune_plan(*P, s);
    if (st != DMUON_OK) return st;
    if (P->ws_bytes > bytes) return fail(DMUON_ERR_WORKSPACE, "internal: the tuned plan needs more workspace");
    if ((e = up(P->off_items, P->items.data(), sizeof(int4) * P->items.size())) != cudaSuccess ||
        (e = cudaMemsetAsync(ws + P->off_status, 0, 4, s)) != cudaSuccess || (e = cudaStreamSynchronize(s)) != cudaSuccess)
      return cuda_fail(e, "tuned table upload");
  }

  // per-launch kernel parameters
  P->tc_params.clear();
  P->simt_params.clear();
  const int4* items = reinterpret_cast<const int4*>(ws + P->off_items);
  for (Launch& L : P->launches) {
    if (L.kind == DMUON_KIND_MOMENTUM || L.kind == DMUON_KIND_UPDATE0) {
      const int per_sm = (L.kind == DMUON_KIND_MOMENTUM) ? momentum_blocks_per_sm(sp.grad_bf16, sp.x_bf16) : 4;
      L.grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(P->n_units, (int64_t)per_sm * P->num_sms)));
      continue;
    }
    if (L.kind == DMUON_KIND_NORM) {  // one CTA per matrix, up to 8 per SM
      L.grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(P->shapes.size(), 8LL * P->num_sms)));
      continue;
    }
    const std::vector<int>& ch = P->chunks[L.chunk];
    const ListRef& lr = (L.list == kListGram)   ? P->gram_lists[L.chunk]
                        : (L.list == kListPoly) ? P->poly_lists[L.chunk]
                                                : P->gemm_lists[L.chunk];
    auto view = [&](const BucketPlan& B, int role) { return view_of(*P, B, role); };
    if (P->tc) {
      TcParams tp;
      std::memset(&tp, 0, sizeof(tp));
      for (size_t lb = 0; lb < ch.size(); ++lb) {
        const BucketPlan& B = P->buckets[ch[lb]];
        // a pair's CTAs each load 128 rows of a K-major B operand
        if (test_hook("bind_maps")) return fail(DMUON_ERR_CUDA, "injected failure (DMUON_TEST_FAIL=bind_maps)");
        dmuon_status st = fill_tc_bucket(*P, B, L.phase, L.pair ? 128 : L.bn, L.opA, L.opB, L.out, L.aux, tp.bk[lb]);
        if (st != DMUON_OK) return st;
      }
      tp.items = items + lr.first;
      tp.n_items = lr.count;
      tp.first = L.first;
      tp.last = L.last;
      tp.a = L.a;
      tp.b = L.b;
      tp.c = L.c;
      tp.diag = L.diag;
      tp.mats = sp.mats;
      tp.ptrs = sp.ptrs;
      tp.s_norm = sp.s_norm;
      tp.capture = sp.capture;
      tp.status = sp.status;
      tp.param_bf16 = sp.param_bf16;
      tp.timeout_ns = 2000000000LL;
      const size_t li = static_cast<size_t>(&L - P->launches.data());
      tp.sched = (P->flags & DMUON_FLAG_STATIC_TILES)
                     ? nullptr
                     : reinterpret_cast<unsigned*>(ws + P->off_sched + kSchedBytes * static_cast<int64_t>(li));
      L.grid = L.pair ? std::max(1, std::min(lr.count, P->num_sms / 2)) : std::max(1, std::min(lr.count, P->num_sms));
      L.param_index = static_cast<int>(P->tc_params.size());
      P->tc_params.push_back(tp);
    } else {
      SimtParams sm;
      std::memset(&sm, 0, sizeof(sm));
      for (size_t lb = 0; lb < ch.size(); ++lb) {
        const BucketPlan& B = P->buckets[ch[lb]];
        SimtBucket& sb = sm.bk[lb];
        sb.slot_mat = reinterpret_cast<const int32_t*>(ws + B.off_slotmat);
        sb.m = B.m;
        sb.n = B.n;
        const View va = view(B, L.opA), vb = view(B, L.opB), vo = view(B, L.out), vx = view(B, L.aux);
        sb.opA = reinterpret_cast<const float*>(va.base);
        sb.a_mat_stride = va.mat_bytes / 4;
        sb.a_ld = va.ld;
        sb.opB = reinterpret_cast<const float*>(vb.base);
        sb.b_mat_stride = vb.mat_bytes / 4;
        sb.b_ld = vb.ld;
        sb.out = reinterpret_cast<float*>(vo.base);
        sb.out_mat_stride = vo.mat_bytes / 4;
        sb.out_ld = vo.ld;
        sb.aux = reinterpret_cast<const float*>(vx.base);
        sb.aux_mat_stride = vx.mat_bytes / 4;
        sb.aux_ld = vx.ld;
        sb.kdim = (L.phase == kPhaseGemm) ? B.m : va.inner;
      }
      sm.items = items + lr.first;
      sm.n_items = lr.count;
      sm.first = L.first;
      sm.last = L.last;
      sm.a = L.a;
      sm.b = L.b;
      sm.c = L.c;
      sm.diag = L.diag;
      sm.mats = sp.mats;
      sm.ptrs = sp.ptrs;
      sm.s_norm = sp.s_norm;
      sm.capture = sp.capture;
      sm.param_bf16 = sp.param_bf16;
      L.grid = std::max(1, lr.count);
      L.param_index = static_cast<int>(P->simt_params.size());
      P->simt_params.push_back(sm);
    }
  }

  // pinned staging for the per-step pointer tables
  if (test_hook("bind_staging")) return fail(DMUON_ERR_CUDA, "injected failure (DMUON_TEST_FAIL=bind_staging)");
  if (P->host_ptrs == nullptr && (e = cudaMallocHost(&P->host_ptrs, 8 * 3 * P->mats.size() * kPtrSlots)) != cudaSuccess)
    return cuda_fail(e, "cudaMallocHost");
  if (P->host_status == nullptr) {
    void* hs = nullptr;
    if ((e = cudaHostAlloc(&hs, 64, cudaHostAllocMapped)) != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
    P->host_status = static_cast<unsigned*>(hs);
  }
  {  // its device address in this (possibly new) device's context
    void* dp = nullptr;
    if ((e = cudaHostGetDevicePointer(&dp, P->host_status, 0)) != cudaSuccess)
      return cuda_fail(e, "cudaHostGetDevicePointer");
    P->host_status_dev = static_cast<unsigned*>(dp);
  }
  if (P->off_wmaps >= 0 && P->host_wmaps == nullptr &&
      (e = cudaMallocHost(&P->host_wmaps, sizeof(CUtensorMap) * P->mats.size() * kPtrSlots)) != cudaSuccess)
    return cuda_fail(e, "cudaMallocHost");
  for (int k = 0; k < kPtrSlots; ++k)
    if (P->ptr_event[k] == nullptr &&
        (e = cudaEventCreateWithFlags(&P->ptr_event[k], cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "cudaEventCreate");
  for (int k = 0; k < kPtrSlots; ++k) {
    P->slot_ptrs[k].clear();
    P->slot_stamp[k] = 0;
  }
  unbind.done = true;
  logf("bind %p: device %d, %d SMs, workspace %p (%zu bytes)%s", (void*)P, P->device, P->num_sms, (void*)P->ws,
       bytes, P->tuned ? ", tuned" : "");
  return DMUON_OK;
}

dmuon_status dmuon_step(dmuon_plan_t P, void* const* params, const void* const* grads, void* const* momenta,
                        float lr, float mu, int32_t nesterov, void* stream) {
  g_err.clear();
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "plan is NULL");
  if (P->ws == nullptr) return fail(DMUON_ERR_NOT_BOUND, "plan has no workspace (call dmuon_plan_bind)");
  if (params == nullptr || grads == nullptr || momenta == nullptr)
    return fail(DMUON_ERR_INVALID_ARG, "pointer array is NULL");
  if (!std::isfinite(lr) || !std::isfinite(mu)) return fail(DMUON_ERR_INVALID_ARG, "lr and mu must be finite");
  if (nesterov != 0 && nesterov != 1) return fail(DMUON_ERR_INVALID_ARG, "nesterov must be 0 or 1");
  int dev = -1;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != P->device) return fail(DMUON_ERR_INVALID_ARG, "current device %d is not the bound device %d", dev,
                                    P->device);
  const size_t n = P->mats.size();
  std::vector<uint64_t> cur(3 * n);
  for (size_t i = 0; i < n; ++i) {
    const uint64_t w = reinterpret_cast<uint64_t>(params[i]), g = reinterpret_cast<uint64_t>(grads[i]),
                   m = reinterpret_cast<uint64_t>(momenta[i]);
    if (w == 0 || g == 0 || m == 0) return fail(DMUON_ERR_INVALID_ARG, "matrix %zu has a NULL pointer", i);
    if ((w | g | m) & 15) return fail(DMUON_ERR_INVALID_ARG, "matrix %zu: pointers must be 16-byte aligned", i);
    cur[i] = w;
    cur[n + i] = g;
    cur[2 * n + i] = m;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // a resident table with these pointers, else refill the least recently used slot (the copy is
  // ordered on the stream after every earlier step that may still read that slot)
  int slot = -1;
  for (int k = 0; k < kPtrSlots && slot < 0; ++k)
    if (P->slot_ptrs[k] == cur) slot = k;
  const size_t tab = cur.size();
  if (slot < 0) {
    slot = 0;
    for (int k = 1; k < kPtrSlots; ++k)
      if (P->slot_stamp[k] < P->slot_stamp[slot]) slot = k;
    if (P->ptr_event_pending[slot]) {
      if ((e = cudaEventSynchronize(P->ptr_event[slot])) != cudaSuccess)
        return cuda_fail(e, "cudaEventSynchronize");
      P->ptr_event_pending[slot] = false;
    }
    P->slot_ptrs[slot].clear();  // holds no valid set until both uploads below are queued
    if (P->off_wmaps >= 0) {
      CUtensorMap* wst = P->host_wmaps + slot * n;
      for (size_t i = 0; i < n; ++i) {
        dmuon_status st = make_wmap(wst + i, params[i], P->mats[i].rows, P->mats[i].cols);
        if (st != DMUON_OK) return st;
      }
      if ((e = cudaMemcpyAsync(P->ws + P->off_wmaps + sizeof(CUtensorMap) * n * slot, wst, sizeof(CUtensorMap) * n,
                               cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "weight tensor-map upload");
    }
    uint64_t* stage = P->host_ptrs + slot * tab;
    std::memcpy(stage, cur.data(), 8 * tab);
    if ((e = cudaMemcpyAsync(P->ws + P->off_ptrs + 8 * tab * slot, stage, 8 * tab, cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
      return cuda_fail(e, "pointer table upload");
    if ((e = cudaEventRecord(P->ptr_event[slot], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    P->ptr_event_pending[slot] = true;
    P->slot_ptrs[slot] = std::move(cur);
  }
  P->slot_stamp[slot] = ++P->ptr_clock;
  const uint64_t* dptrs = reinterpret_cast<const uint64_t*>(P->ws + P->off_ptrs + 8 * tab * slot);
  const CUtensorMap* dwmaps =
      P->off_wmaps >= 0 ? reinterpret_cast<const CUtensorMap*>(P->ws + P->off_wmaps + sizeof(CUtensorMap) * n * slot)
                        : nullptr;

  StreamParams sp = P->sp;
  sp.mu = mu;
  sp.lr = lr;
  sp.nesterov = nesterov;
  sp.ptrs = dptrs;
  if (P->steps_taken++ == 0)
    logf("step: plan %p, first step: %zu launches, pointer slot %d, lr %g mu %g nesterov %d", (void*)P,
         P->launches.size(), slot, lr, mu, nesterov);
  struct NvtxStep {
    NvtxStep() { nvtxRangePushA("dmuon_step"); }
    ~NvtxStep() { nvtxRangePop(); }
  } nvtx_step;
  for (size_t li = 0; li < P->launches.size(); ++li) {
    const Launch& L = P->launches[li];
    struct NvtxLaunch {
      explicit NvtxLaunch(int kind) { nvtxRangePushA(kind_range_name(kind)); }
      ~NvtxLaunch() { nvtxRangePop(); }
    } nvtx_launch(L.kind);
    if (static_cast<int>(li) == P->first_w_launch && P->w_wait != nullptr &&
        (e = cudaStreamWaitEvent(s, P->w_wait, 0)) != cudaSuccess)
      return cuda_fail(e, "cudaStreamWaitEvent (weight events)");
    std::vector<DbgSample> dbg;
    const bool debug = (P->flags & DMUON_FLAG_DEBUG_CHECKS) != 0;
    if (debug) {
      dmuon_status sd = debug_before(*P, L, static_cast<int>(li), params, grads, momenta, dbg, s);
      if (sd != DMUON_OK) return sd;
    }
    dmuon_status st = record_launch(*P, L, s, true);
    if (st != DMUON_OK) return st;
    if (debug && test_skip_launch(static_cast<int>(li))) {
      // test hook (debug mode only): the launch is left out, so its outputs keep what was there
      e = cudaSuccess;
    } else if (L.kind == DMUON_KIND_MOMENTUM) {
      e = launch_momentum(sp, L.grid, s);
    } else if (L.kind == DMUON_KIND_NORM) {
      e = launch_norm_finalize(sp, L.grid, s);
    } else if (L.kind == DMUON_KIND_UPDATE0) {
      e = launch_update0(sp, L.grid, s);
    } else if (P->tc) {
      TcParams& tp = P->tc_params[L.param_index];
      tp.lr = lr;
      tp.ptrs = dptrs;
      tp.wmaps = dwmaps;
      tp.cta_times = P->cta_times ? reinterpret_cast<unsigned long long*>(P->ws + P->off_cta) +
                                        2LL * kMaxCtaRecords * static_cast<int64_t>(li)
                                  : nullptr;
      e = L.pair ? launch_tc_pair(L.phase, tp, L.grid, s) : launch_tc(L.phase, L.bn, tp, L.grid, s);
    } else {
      SimtParams& p = P->simt_params[L.param_index];
      p.lr = lr;
      p.ptrs = dptrs;
      e = launch_simt(L.phase, p, L.grid, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    ++P->launch_count;
    st = record_launch(*P, L, s, false);
    if (st != DMUON_OK) return st;
    if (debug) {
      st = debug_after(*P, L, static_cast<int>(li), params, momenta, dbg, lr, mu, nesterov, s);
      if (st != DMUON_OK) return st;
    }
    if (static_cast<int>(li) == P->last_w_launch && P->w_done != nullptr &&
        (e = cudaEventRecord(P->w_done, s)) != cudaSuccess)
      return cuda_fail(e, "cudaEventRecord (weight events)");
  }
  return DMUON_OK;
}

dmuon_status dmuon_set_weight_events(dmuon_plan_t P, void* wait_before_write, void* after_write) {
  g_err.clear();
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "plan is NULL");
  P->w_wait = reinterpret_cast<cudaEvent_t>(wait_before_write);
  P->w_done = reinterpret_cast<cudaEvent_t>(after_write);
  return DMUON_OK;
}

dmuon_status dmuon_read_device_status(dmuon_plan_t P, void* stream, uint32_t* bits) {
  if (P == nullptr || bits == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (P->ws == nullptr) return fail(DMUON_ERR_NOT_BOUND, "plan is not bound");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  // a one-thread kernel moves the word into mapped host memory and clears it (no copy engine, so
  // the read does not wait behind other streams' transfers)
  *reinterpret_cast<volatile unsigned*>(P->host_status) = 0u;
  if ((e = launch_status_readout(reinterpret_cast<unsigned*>(P->ws + P->off_status), P->host_status_dev, s)) !=
      cudaSuccess)
    return cuda_fail(e, "status readout launch");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "status sync");
  *bits = *reinterpret_cast<volatile unsigned*>(P->host_status);
  return DMUON_OK;
}

dmuon_status dmuon_read_update(dmuon_plan_t P, int32_t mat, float* d_dst, void* stream) {
  if (P == nullptr || d_dst == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (!(P->flags & DMUON_FLAG_CAPTURE_UPDATE))
    return fail(DMUON_ERR_UNSUPPORTED, "plan was made without DMUON_FLAG_CAPTURE_UPDATE");
  if (P->ws == nullptr) return fail(DMUON_ERR_NOT_BOUND, "plan is not bound");
  if (mat < 0 || mat >= static_cast<int32_t>(P->mats.size()))
    return fail(DMUON_ERR_INVALID_ARG, "matrix index %d out of range", mat);
  const MatDev& d = P->mats[mat];
  cudaError_t e = cudaMemcpyAsync(d_dst, P->ws + P->off_capture + 4 * d.cap_off, 4LL * d.rows * d.cols,
                                  cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DMUON_OK : cuda_fail(e, "update copy");
}

dmuon_status dmuon_plan_describe(dmuon_plan_t P, char* buf, size_t len, size_t* needed) {
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "plan is NULL");
  std::string j = "{";
  char t[512];
  snprintf(t, sizeof t,
           "\"n_mats\": %zu, \"ns_steps\": %d, \"compute\": \"%s\", \"tile\": [%d, %d], \"workspace_bytes\": %zu, "
           "\"stream_units\": %lld, \"chunks\": %zu, \"tuned\": %s, \"tune_timed_buckets\": %d, "
           "\"tune_cached_buckets\": %d, ",
           P->mats.size(), P->ns_steps, P->tc ? "bf16" : "f32", P->tile_m, P->tile_n, P->ws_bytes,
           (long long)P->n_units, P->chunks.size(), P->tuned ? "true" : "false", P->tune_timed, P->tune_cached);
  j += t;
  j += "\"buckets\": [";
  for (size_t b = 0; b < P->buckets.size(); ++b) {
    const BucketPlan& B = P->buckets[b];
    snprintf(t, sizeof t,
             "%s{\"m\": %d, \"n\": %d, \"count\": %d, \"transposed\": %d, \"x_ld\": %d, \"m_ld\": %d, "
             "\"form\": \"%s\", \"pair\": %s, \"bn_sym\": %d, \"bn_gemm\": %d, "
             "\"tile_ms\": [%.6g, %.6g, %.6g], \"tune_cost\": [%.6g, %.6g, %.6g], "
             "\"tune_cost_gemm\": [%.6g, %.6g, %.6g]}",
             b ? ", " : "", B.m, B.n, B.count, B.n_transposed, B.x_ld, B.m_ld, B.gram ? "gram" : "standard",
             B.pair ? "true" : "false", B.bn_sym, B.bn_gemm, B.tile_ms[0], B.tile_ms[1], B.tile_ms[2],
             B.tune_cost[0], B.tune_cost[1], B.tune_cost[2], B.tune_gemm[0], B.tune_gemm[1], B.tune_gemm[2]);
    j += t;
  }
  j += "], \"regions\": {";
  // Workspace byte ranges [offset, bytes]: "tables" are written by bind and only read by steps;
  // "scratch" is written by every step before the step reads it (per-matrix s, partial sums,
  // the bucket buffers, the update capture); "status" accumulates device status bits.
  snprintf(t, sizeof t, "\"status\": [%lld, 4], \"tables\": [[%lld, %lld]", (long long)P->off_status,
           (long long)P->off_mats, (long long)(P->off_probe + (int64_t)sizeof(int4) * kProbeTiles - P->off_mats));
  j += t;
  for (const BucketPlan& B : P->buckets) {
    snprintf(t, sizeof t, ", [%lld, %lld]", (long long)B.off_slotmat, 4LL * B.count);
    j += t;
  }
  snprintf(t, sizeof t, "], \"scratch\": [[%lld, %lld], [%lld, %lld]", (long long)P->off_s, 4LL * (long long)P->mats.size(),
           (long long)P->off_partial, (long long)(4LL * kPartialsPerUnit * std::max<int64_t>(P->n_units, 1)));
  j += t;
  for (const BucketPlan& B : P->buckets)
    for (int r = 0; r < kBufCount; ++r)
      if (B.off[r] >= 0) {
        snprintf(t, sizeof t, ", [%lld, %lld]", (long long)B.off[r],
                 (long long)((B.is_x(r) ? B.x_mat_bytes : B.a_mat_bytes) * B.count));
        j += t;
      }
  if (P->off_capture >= 0) {
    snprintf(t, sizeof t, ", [%lld, %lld]", (long long)P->off_capture, 4LL * std::max<int64_t>(P->cap_elems, 1));
    j += t;
  }
  j += "]}";
  j += ", \"lists\": [";
  for (size_t c = 0; c < P->gram_lists.size(); ++c) {
    snprintf(t, sizeof t, "%s{\"chunk\": %zu, \"gram\": %d, \"poly\": %d, \"gemm\": %d}", c ? ", " : "", c,
             P->gram_lists[c].count, P->poly_lists[c].count, P->gemm_lists[c].count);
    j += t;
  }
  j += "], \"launches\": [";
  for (size_t l = 0; l < P->launches.size(); ++l) {
    const Launch& L = P->launches[l];
    snprintf(t, sizeof t,
             "%s{\"kind\": %d, \"step\": %d, \"chunk\": %d, \"bn\": %d, \"pair\": %s, \"grid\": %d, "
             "\"work\": %.17g, \"a\": %.9g, \"b\": %.9g, \"c\": %.9g, \"diag\": %.9g}",
             l ? ", " : "", L.kind, L.step, L.chunk, L.bn, L.pair ? "true" : "false", L.grid, L.work, L.a, L.b,
             L.c, L.diag);
    j += t;
  }
  j += "]}";
  if (needed) *needed = j.size() + 1;
  if (buf != nullptr && len > 0) {
    const size_t k = std::min(len - 1, j.size());
    std::memcpy(buf, j.data(), k);
    buf[k] = '\0';
  }
  return DMUON_OK;
}

dmuon_status dmuon_profile_begin(dmuon_plan_t P, int32_t max_launches) {
  if (P == nullptr || max_launches <= 0 || max_launches > (1 << 20))
    return fail(DMUON_ERR_INVALID_ARG, "bad profile arguments");
  destroy_events(*P);
  P->ev_start.resize(max_launches);
  P->ev_stop.resize(max_launches);
  for (int i = 0; i < max_launches; ++i) {
    cudaError_t e1 = cudaEventCreate(&P->ev_start[i]), e2 = cudaEventCreate(&P->ev_stop[i]);
    if (e1 != cudaSuccess || e2 != cudaSuccess) {
      P->ev_start.resize(i);
      P->ev_stop.resize(i);
      destroy_events(*P);
      return cuda_fail(e1 != cudaSuccess ? e1 : e2, "cudaEventCreate");
    }
  }
  P->prof_kind.assign(max_launches, 0);
  P->prof_work.assign(max_launches, 0.0);
  P->prof_max = max_launches;
  P->prof_n = 0;
  P->prof = true;
  return DMUON_OK;
}

dmuon_status dmuon_profile_end(dmuon_plan_t P, int32_t* kinds, float* ms, double* work, int32_t cap,
                               int32_t* n) {
  if (P == nullptr || n == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (!P->prof) return fail(DMUON_ERR_INVALID_ARG, "profiling was not started");
  *n = P->prof_n;
  for (int i = 0; i < P->prof_n && i < cap; ++i) {
    cudaError_t e = cudaEventSynchronize(P->ev_stop[i]);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, P->ev_start[i], P->ev_stop[i]);
    if (e != cudaSuccess) {
      destroy_events(*P);
      return cuda_fail(e, "profile events");
    }
    if (kinds) kinds[i] = P->prof_kind[i];
    if (ms) ms[i] = t;
    if (work) work[i] = P->prof_work[i];
  }
  destroy_events(*P);
  return DMUON_OK;
}

dmuon_status dmuon_plan_costs(dmuon_plan_t P, double* per_matrix_ms, int32_t n) {
  if (P == nullptr || per_matrix_ms == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (n != static_cast<int32_t>(P->mats.size())) return fail(DMUON_ERR_INVALID_ARG, "n must equal the plan's n_mats");
  if (!P->tuned) return fail(DMUON_ERR_UNSUPPORTED, "the plan was not tuned (bind it with DMUON_FLAG_TUNE)");
  const double S = P->ns_steps;
  std::vector<int4> t;
  std::vector<double> per_bucket(P->buckets.size());
  for (size_t b = 0; b < P->buckets.size(); ++b) {
    BucketPlan B = P->buckets[b];
    B.count = 1;
    t.clear();
    add_tiles(*P, DMUON_KIND_GRAM, 0, B, t);
    const double nsym = static_cast<double>(t.size());
    t.clear();
    add_tiles(*P, DMUON_KIND_GEMM, 0, B, t);
    const double ngemm = static_cast<double>(t.size());
    const double n_xx = B.gram ? 1.0 : S, n_mm = B.gram ? 4.0 * S - 3.0 : S, n_gm = B.gram ? 1.0 : S;
    // time one SM spends on the matrix, spread over all SMs
    per_bucket[b] = (nsym * (n_xx * B.tile_ms[0] + n_mm * B.tile_ms[1]) + ngemm * n_gm * B.tile_ms[2]) / P->num_sms;
  }
  for (size_t i = 0; i < P->mats.size(); ++i) per_matrix_ms[i] = per_bucket[P->mats[i].bucket];
  return DMUON_OK;
}

dmuon_status dmuon_profile_cta_times(dmuon_plan_t P, int32_t enable) {
  if (P == nullptr) return fail(DMUON_ERR_INVALID_ARG, "plan is NULL");
  P->cta_times = enable != 0;
  return DMUON_OK;
}

dmuon_status dmuon_read_cta_times(dmuon_plan_t P, int32_t launch, uint64_t* out, int32_t cap, int32_t* n_ctas,
                                  void* stream) {
  if (P == nullptr || n_ctas == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (P->ws == nullptr) return fail(DMUON_ERR_NOT_BOUND, "plan is not bound");
  if (launch < 0 || launch >= static_cast<int32_t>(P->launches.size()))
    return fail(DMUON_ERR_INVALID_ARG, "launch index %d out of range", launch);
  const Launch& L = P->launches[launch];
  const bool tc_kind = L.kind == DMUON_KIND_GRAM || L.kind == DMUON_KIND_POLY || L.kind == DMUON_KIND_GEMM ||
                       L.kind == DMUON_KIND_SYMM;
  if (!P->tc || !tc_kind) {
    *n_ctas = 0;
    return DMUON_OK;
  }
  const int n = std::min<int>(L.pair ? 2 * L.grid : L.grid, kMaxCtaRecords);  // a pair launch's grid counts pairs
  *n_ctas = n;
  if (out == nullptr || cap <= 0) return DMUON_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const size_t bytes = 16ULL * std::min(n, cap);
  if ((e = cudaMemcpyAsync(out, P->ws + P->off_cta + 16LL * kMaxCtaRecords * launch, bytes, cudaMemcpyDeviceToHost,
                           s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess)
    return cuda_fail(e, "per-CTA times copy");
  return DMUON_OK;
}

dmuon_status dmuon_launch_count(dmuon_plan_t P, int64_t* count) {
  if (P == nullptr || count == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  *count = P->launch_count;
  return DMUON_OK;
}

dmuon_status dmuon_selftest_wait_timeout(void* d_scratch, int64_t limit_ns, void* stream, uint32_t* bits) {
  if (d_scratch == nullptr || bits == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (limit_ns < 1000000LL || limit_ns > 5000000000LL)
    return fail(DMUON_ERR_INVALID_ARG, "limit_ns must be in 1e6..5e9");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* st = static_cast<unsigned*>(d_scratch);
  cudaError_t e;
  if ((e = cudaMemsetAsync(st, 0, 4, s)) != cudaSuccess) return cuda_fail(e, "memset");
  if ((e = launch_wait_timeout_selftest(st, limit_ns, s)) != cudaSuccess) return cuda_fail(e, "launch");
  uint32_t v = 0;
  if ((e = cudaMemcpyAsync(&v, st, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess) return cuda_fail(e, "copy");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "sync");
  *bits = v;
  return DMUON_OK;
}

void dmuon_plan_destroy(dmuon_plan_t P) {
  if (P == nullptr) return;
  destroy_events(*P);
  for (int k = 0; k < kPtrSlots; ++k) {
    if (P->ptr_event[k]) {
      cudaEventSynchronize(P->ptr_event[k]);
      cudaEventDestroy(P->ptr_event[k]);
    }
  }
  if (P->host_ptrs) cudaFreeHost(P->host_ptrs);
  if (P->host_wmaps) cudaFreeHost(P->host_wmaps);
  if (P->host_status) cudaFreeHost(P->host_status);
  delete P;
}

}  // extern "C"
