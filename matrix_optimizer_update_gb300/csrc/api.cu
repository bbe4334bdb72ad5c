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
// tiles are sorted by cost, largest first, and dealt round-robin to the
// persistent CTAs: the greedy fallback of the cost-based balancing of
// section 2.3, applied to SMs instead of owner ranks.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "dmuon.h"
#include "internal.h"

using namespace dmuon;

namespace {

thread_local std::string g_err;

dmuon_status fail(dmuon_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

dmuon_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DMUON_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kAlign = 1024;
int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct BucketPlan {
  int32_t m = 0, n = 0, count = 0, n_transposed = 0;
  int32_t x_ld = 0, m_ld = 0;
  std::vector<int32_t> mats;  // slot -> global matrix index
  int64_t off_slotmat = -1;
  int64_t off_x[2] = {-1, -1}, off_a = -1, off_b = -1;
  int64_t x_mat_bytes = 0, a_mat_bytes = 0;
};

struct ListRef {
  int64_t first = 0;  // index into items
  int32_t count = 0;
};

struct Launch {
  int kind = 0;   // DMUON_KIND_*
  int step = -1;  // Newton-Schulz step
  int chunk = 0;
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
  std::vector<int4> items;
  std::vector<ListRef> gram_lists, poly_lists, gemm_lists;
  std::vector<Launch> launches;
  // ---- workspace layout (byte offsets)
  size_t ws_bytes = 0;
  int64_t off_status = 0, off_counters = 0, off_s = 0, off_partial = 0, off_mats = 0, off_ub = 0, off_ptrs = 0,
          off_items = 0, off_capture = -1;
  int64_t cap_elems = 0;
  // ---- binding
  char* ws = nullptr;
  int device = -1;
  int num_sms = 0;
  StreamParams sp{};
  std::vector<TcParams> tc_params;
  std::vector<SimtParams> simt_params;
  uint64_t* host_ptrs = nullptr;  // pinned staging of the pointer table
  std::vector<uint64_t> last_ptrs;
  cudaEvent_t ptr_event = nullptr;
  bool ptr_event_pending = false;
  // ---- profiling
  bool prof = false;
  int32_t prof_max = 0, prof_n = 0;
  std::vector<cudaEvent_t> ev_start, ev_stop;
  std::vector<int32_t> prof_kind;
  std::vector<double> prof_work;
  int64_t launch_count = 0;
};

namespace {

double phase_flops(int kind, double m, double n) {
  switch (kind) {
    case DMUON_KIND_GRAM:
      return m * (m + 1) * n;
    case DMUON_KIND_POLY:
      return m * m * (m + 1);
    case DMUON_KIND_GEMM:
      return 2 * m * m * n;
    default:
      return 0;
  }
}

int dtype_bytes(int32_t d) { return d == DMUON_BF16 ? 2 : 4; }

// Tiles of one phase for one bucket, appended in cost order.
void add_tiles(const dmuon_plan_s& P, int kind, int bucket_local, const BucketPlan& B, std::vector<int4>& out) {
  const int BM = P.tile_m, BN = P.tile_n;
  const int tm = static_cast<int>(cdiv(B.m, BM));
  if (kind == DMUON_KIND_GEMM) {
    const int tn = static_cast<int>(cdiv(B.n, BN));
    for (int s = 0; s < B.count; ++s)
      for (int tj = 0; tj < tn; ++tj)
        for (int ti = 0; ti < tm; ++ti) out.push_back(make_int4(bucket_local, s, ti, tj));
  } else {
    const int tn = static_cast<int>(cdiv(B.m, BN));
    for (int s = 0; s < B.count; ++s)
      for (int ti = 0; ti < tm; ++ti)
        for (int tj = 0; tj < tn; ++tj)
          if (tj * BN + BN - 1 >= ti * BM) out.push_back(make_int4(bucket_local, s, ti, tj));
  }
}

dmuon_status build_plan(dmuon_plan_s& P) {
  const int n_mats = static_cast<int>(P.shapes.size());
  P.tc = (P.dt.compute == DMUON_BF16);
  P.xel = P.tc ? 2 : 4;
  P.tile_m = P.tc ? kTcBM : kSimtBM;
  P.tile_n = P.tc ? kTcBN : kSimtBN;
  const int ld_mult = P.tc ? 8 : 4;

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
    P.buckets[b].m_ld = static_cast<int32_t>(align_up(order[b].first, ld_mult));
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
    d.flat = (!d.transposed && c % 8 == 0) ? 1 : 0;
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

  // ---- launch chunks of at most kMaxBucketsPerLaunch buckets
  P.chunks.clear();
  for (size_t b = 0; b < P.buckets.size(); b += kMaxBucketsPerLaunch) {
    std::vector<int> ch;
    for (size_t q = b; q < std::min(P.buckets.size(), b + kMaxBucketsPerLaunch); ++q) ch.push_back((int)q);
    P.chunks.push_back(ch);
  }

  // ---- cost-ordered tile lists per (phase, chunk)
  P.items.clear();
  auto build_list = [&](int kind, const std::vector<int>& ch) {
    std::vector<std::pair<double, int4>> tmp;
    for (size_t lb = 0; lb < ch.size(); ++lb) {
      const BucketPlan& B = P.buckets[ch[lb]];
      std::vector<int4> t;
      add_tiles(P, kind, static_cast<int>(lb), B, t);
      const double cost = (kind == DMUON_KIND_GRAM) ? B.n : B.m;  // K extent of every tile
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
  P.off_counters = take(4LL * n_mats);
  P.off_s = take(4LL * n_mats);
  P.off_partial = take(4LL * std::max<int64_t>(units, 1));
  P.off_mats = take((int64_t)sizeof(MatDev) * n_mats);
  P.off_ub = take(8LL * (n_mats + 1));
  P.off_ptrs = take(8LL * 3 * n_mats);
  P.off_items = take((int64_t)sizeof(int4) * std::max<size_t>(P.items.size(), 1));
  for (BucketPlan& B : P.buckets) {
    B.off_slotmat = take(4LL * B.count);
    B.x_mat_bytes = (int64_t)B.m * B.x_ld * P.xel;
    B.a_mat_bytes = (int64_t)B.m * B.m_ld * P.xel;
    B.off_x[0] = take(B.x_mat_bytes * B.count);
    B.off_x[1] = (P.ns_steps >= 2) ? take(B.x_mat_bytes * B.count) : -1;
    if (P.ns_steps >= 1) {
      B.off_a = take(B.a_mat_bytes * B.count);
      B.off_b = take(B.a_mat_bytes * B.count);
    }
  }
  for (int i = 0; i < n_mats; ++i) {
    const BucketPlan& B = P.buckets[P.mats[i].bucket];
    P.mats[i].x0_off = B.off_x[0] + (int64_t)P.mats[i].slot * B.x_mat_bytes;
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
  if (P.ns_steps == 0) {
    Launch u;
    u.kind = DMUON_KIND_UPDATE0;
    u.work = elems * (2 * pb + P.xel);
    P.launches.push_back(u);
  }
  for (int k = 0; k < P.ns_steps; ++k) {
    for (int kind : {DMUON_KIND_GRAM, DMUON_KIND_POLY, DMUON_KIND_GEMM}) {
      for (size_t c = 0; c < P.chunks.size(); ++c) {
        Launch x;
        x.kind = kind;
        x.step = k;
        x.chunk = static_cast<int>(c);
        for (int b : P.chunks[c]) {
          const BucketPlan& B = P.buckets[b];
          x.work += B.count * phase_flops(kind, B.m, B.n);
        }
        P.launches.push_back(x);
      }
    }
  }
  return DMUON_OK;
}

dmuon_status make_map(CUtensorMap* map, const void* base, int inner, int rows, int count, int ld_elems,
                      int box_inner, int box_rows) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)ld_elems * 2, (cuuint64_t)ld_elems * 2 * rows};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
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
  if (flags & ~DMUON_FLAG_CAPTURE_UPDATE) return fail(DMUON_ERR_UNSUPPORTED, "unknown flag bits 0x%x", flags);
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
  if (d_workspace == nullptr) return fail(DMUON_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(d_workspace) % kAlign != 0)
    return fail(DMUON_ERR_WORKSPACE, "workspace must be %lld-byte aligned", (long long)kAlign);
  if (bytes < P->ws_bytes)
    return fail(DMUON_ERR_WORKSPACE, "workspace has %zu bytes, plan needs %zu", bytes, P->ws_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaGetDevice(&P->device)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if ((e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, d_workspace) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return fail(DMUON_ERR_WORKSPACE, "workspace is not device memory");
  }
  if (P->tc) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, P->device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, P->device);
    if (major != 10 || minor != 3)
      return fail(DMUON_ERR_UNSUPPORTED, "bf16 compute needs an sm_103 GPU (found sm_%d%d)", major, minor);
  }
  P->ws = static_cast<char*>(d_workspace);
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
  if ((e = cudaMemsetAsync(ws + P->off_status, 0, P->off_s - P->off_status, s)) != cudaSuccess)
    return cuda_fail(e, "cudaMemsetAsync");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "bind sync");

  // momentum-pass parameters
  StreamParams& sp = P->sp;
  sp = StreamParams{};
  sp.mats = reinterpret_cast<const MatDev*>(ws + P->off_mats);
  sp.unit_begin = reinterpret_cast<const int64_t*>(ws + P->off_ub);
  sp.ptrs = reinterpret_cast<const uint64_t*>(ws + P->off_ptrs);
  sp.ws = ws;
  sp.partial = reinterpret_cast<float*>(ws + P->off_partial);
  sp.counters = reinterpret_cast<unsigned*>(ws + P->off_counters);
  sp.s_norm = reinterpret_cast<float*>(ws + P->off_s);
  sp.status = reinterpret_cast<unsigned*>(ws + P->off_status);
  sp.capture = P->off_capture >= 0 ? reinterpret_cast<float*>(ws + P->off_capture) : nullptr;
  sp.n_units = P->n_units;
  sp.n_mats = static_cast<int32_t>(P->mats.size());
  sp.eps = P->eps;
  sp.grad_bf16 = P->dt.grad == DMUON_BF16;
  sp.x_bf16 = P->tc;
  sp.param_bf16 = P->dt.param == DMUON_BF16;

  // per-launch kernel parameters
  P->tc_params.clear();
  P->simt_params.clear();
  const int4* items = reinterpret_cast<const int4*>(ws + P->off_items);
  for (Launch& L : P->launches) {
    if (L.kind == DMUON_KIND_MOMENTUM || L.kind == DMUON_KIND_UPDATE0) {
      L.grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(P->n_units, 4LL * P->num_sms)));
      continue;
    }
    const int k = L.step;
    const std::vector<int>& ch = P->chunks[L.chunk];
    const ListRef& lr = (L.kind == DMUON_KIND_GRAM)   ? P->gram_lists[L.chunk]
                        : (L.kind == DMUON_KIND_POLY) ? P->poly_lists[L.chunk]
                                                      : P->gemm_lists[L.chunk];
    const int xin = k & 1, xout = (k + 1) & 1;
    const bool first = (k == 0), last = (k == P->ns_steps - 1);
    const float a = P->coeffs[3 * k], b = P->coeffs[3 * k + 1], c = P->coeffs[3 * k + 2];
    if (P->tc) {
      TcParams tp;
      std::memset(&tp, 0, sizeof(tp));
      for (size_t lb = 0; lb < ch.size(); ++lb) {
        const BucketPlan& B = P->buckets[ch[lb]];
        TcBucket& tb = tp.bk[lb];
        tb.slot_mat = reinterpret_cast<const int32_t*>(ws + B.off_slotmat);
        tb.m = B.m;
        tb.n = B.n;
        const char* X = ws + B.off_x[xin];
        const char* A = ws + B.off_a;
        const char* Bp = ws + B.off_b;
        dmuon_status st = DMUON_OK;
        if (L.kind == DMUON_KIND_GRAM) {
          st = make_map(&tb.tmA, X, B.n, B.m, B.count, B.x_ld, 64, kTcBM);
          if (st == DMUON_OK) st = make_map(&tb.tmB, X, B.n, B.m, B.count, B.x_ld, 64, kTcBN);
          tb.out = ws + B.off_a;
          tb.out_mat_stride = B.a_mat_bytes;
          tb.out_ld = B.m_ld;
          tb.kdim = B.n;
        } else if (L.kind == DMUON_KIND_POLY) {
          st = make_map(&tb.tmA, A, B.m, B.m, B.count, B.m_ld, 64, kTcBM);
          if (st == DMUON_OK) st = make_map(&tb.tmB, A, B.m, B.m, B.count, B.m_ld, 64, kTcBN);
          tb.out = ws + B.off_b;
          tb.out_mat_stride = B.a_mat_bytes;
          tb.out_ld = B.m_ld;
          tb.aux = A;
          tb.aux_mat_stride = B.a_mat_bytes;
          tb.aux_ld = B.m_ld;
          tb.kdim = B.m;
        } else {
          st = make_map(&tb.tmA, Bp, B.m, B.m, B.count, B.m_ld, 64, kTcBM);
          // X as the MN-major operand: 64 columns (N) x 64 rows (K) per box
          if (st == DMUON_OK) st = make_map(&tb.tmB, X, B.n, B.m, B.count, B.x_ld, 64, 64);
          tb.out = last ? nullptr : ws + B.off_x[xout];
          tb.out_mat_stride = B.x_mat_bytes;
          tb.out_ld = B.x_ld;
          tb.aux = X;
          tb.aux_mat_stride = B.x_mat_bytes;
          tb.aux_ld = B.x_ld;
          tb.kdim = B.m;
        }
        if (st != DMUON_OK) return st;
      }
      tp.items = items + lr.first;
      tp.n_items = lr.count;
      tp.first = first;
      tp.last = last;
      tp.a = a;
      tp.b = b;
      tp.c = c;
      tp.mats = sp.mats;
      tp.ptrs = sp.ptrs;
      tp.s_norm = sp.s_norm;
      tp.capture = sp.capture;
      tp.status = sp.status;
      tp.param_bf16 = sp.param_bf16;
      tp.timeout_ns = 2000000000LL;
      L.grid = std::max(1, std::min(lr.count, P->num_sms));
      L.param_index = static_cast<int>(P->tc_params.size());
      P->tc_params.push_back(tp);
    } else {
      SimtParams p;
      std::memset(&p, 0, sizeof(p));
      for (size_t lb = 0; lb < ch.size(); ++lb) {
        const BucketPlan& B = P->buckets[ch[lb]];
        SimtBucket& sb = p.bk[lb];
        sb.slot_mat = reinterpret_cast<const int32_t*>(ws + B.off_slotmat);
        sb.m = B.m;
        sb.n = B.n;
        const int64_t xs = B.x_mat_bytes / 4, as = B.a_mat_bytes / 4;
        const float* X = reinterpret_cast<const float*>(ws + B.off_x[xin]);
        const float* A = reinterpret_cast<const float*>(ws + B.off_a);
        const float* Bp = reinterpret_cast<const float*>(ws + B.off_b);
        if (L.kind == DMUON_KIND_GRAM) {
          sb.opA = sb.opB = X;
          sb.a_mat_stride = sb.b_mat_stride = xs;
          sb.a_ld = sb.b_ld = B.x_ld;
          sb.out = reinterpret_cast<float*>(ws + B.off_a);
          sb.out_mat_stride = as;
          sb.out_ld = B.m_ld;
          sb.kdim = B.n;
        } else if (L.kind == DMUON_KIND_POLY) {
          sb.opA = sb.opB = A;
          sb.a_mat_stride = sb.b_mat_stride = as;
          sb.a_ld = sb.b_ld = B.m_ld;
          sb.out = reinterpret_cast<float*>(ws + B.off_b);
          sb.out_mat_stride = as;
          sb.out_ld = B.m_ld;
          sb.aux = A;
          sb.aux_mat_stride = as;
          sb.aux_ld = B.m_ld;
          sb.kdim = B.m;
        } else {
          sb.opA = Bp;
          sb.a_mat_stride = as;
          sb.a_ld = B.m_ld;
          sb.opB = X;
          sb.b_mat_stride = xs;
          sb.b_ld = B.x_ld;
          sb.out = last ? nullptr : reinterpret_cast<float*>(ws + B.off_x[xout]);
          sb.out_mat_stride = xs;
          sb.out_ld = B.x_ld;
          sb.aux = X;
          sb.aux_mat_stride = xs;
          sb.aux_ld = B.x_ld;
          sb.kdim = B.m;
        }
      }
      p.items = items + lr.first;
      p.n_items = lr.count;
      p.first = first;
      p.last = last;
      p.a = a;
      p.b = b;
      p.c = c;
      p.mats = sp.mats;
      p.ptrs = sp.ptrs;
      p.s_norm = sp.s_norm;
      p.capture = sp.capture;
      p.param_bf16 = sp.param_bf16;
      L.grid = std::max(1, lr.count);
      L.param_index = static_cast<int>(P->simt_params.size());
      P->simt_params.push_back(p);
    }
  }

  // pinned staging for the per-step pointer table
  if (P->host_ptrs == nullptr) {
    if ((e = cudaMallocHost(&P->host_ptrs, 8 * 3 * P->mats.size())) != cudaSuccess)
      return cuda_fail(e, "cudaMallocHost");
    if ((e = cudaEventCreateWithFlags(&P->ptr_event, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_fail(e, "cudaEventCreate");
  }
  P->last_ptrs.clear();
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
  if (cur != P->last_ptrs) {
    if (P->ptr_event_pending) {
      if ((e = cudaEventSynchronize(P->ptr_event)) != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
      P->ptr_event_pending = false;
    }
    std::memcpy(P->host_ptrs, cur.data(), 8 * cur.size());
    if ((e = cudaMemcpyAsync(P->ws + P->off_ptrs, P->host_ptrs, 8 * cur.size(), cudaMemcpyHostToDevice, s)) !=
        cudaSuccess)
      return cuda_fail(e, "pointer table upload");
    if ((e = cudaEventRecord(P->ptr_event, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    P->ptr_event_pending = true;
    P->last_ptrs = cur;
  }

  StreamParams sp = P->sp;
  sp.mu = mu;
  sp.lr = lr;
  sp.nesterov = nesterov;
  for (const Launch& L : P->launches) {
    dmuon_status st = record_launch(*P, L, s, true);
    if (st != DMUON_OK) return st;
    if (L.kind == DMUON_KIND_MOMENTUM) {
      e = launch_momentum(sp, L.grid, s);
    } else if (L.kind == DMUON_KIND_UPDATE0) {
      e = launch_update0(sp, L.grid, s);
    } else if (P->tc) {
      TcParams& tp = P->tc_params[L.param_index];
      tp.lr = lr;
      e = launch_tc(L.kind, tp, L.grid, s);
    } else {
      SimtParams& p = P->simt_params[L.param_index];
      p.lr = lr;
      e = launch_simt(L.kind, p, L.grid, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    ++P->launch_count;
    st = record_launch(*P, L, s, false);
    if (st != DMUON_OK) return st;
  }
  return DMUON_OK;
}

dmuon_status dmuon_read_device_status(dmuon_plan_t P, void* stream, uint32_t* bits) {
  if (P == nullptr || bits == nullptr) return fail(DMUON_ERR_INVALID_ARG, "NULL argument");
  if (P->ws == nullptr) return fail(DMUON_ERR_NOT_BOUND, "plan is not bound");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(&v, P->ws + P->off_status, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "status read");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "status sync");
  if ((e = cudaMemsetAsync(P->ws + P->off_status, 0, 4, s)) != cudaSuccess) return cuda_fail(e, "status clear");
  *bits = v;
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
           "\"stream_units\": %lld, \"chunks\": %zu, ",
           P->mats.size(), P->ns_steps, P->tc ? "bf16" : "f32", P->tile_m, P->tile_n, P->ws_bytes,
           (long long)P->n_units, P->chunks.size());
  j += t;
  j += "\"buckets\": [";
  for (size_t b = 0; b < P->buckets.size(); ++b) {
    const BucketPlan& B = P->buckets[b];
    snprintf(t, sizeof t, "%s{\"m\": %d, \"n\": %d, \"count\": %d, \"transposed\": %d, \"x_ld\": %d, \"m_ld\": %d}",
             b ? ", " : "", B.m, B.n, B.count, B.n_transposed, B.x_ld, B.m_ld);
    j += t;
  }
  j += "], \"lists\": [";
  for (size_t c = 0; c < P->gram_lists.size(); ++c) {
    snprintf(t, sizeof t, "%s{\"chunk\": %zu, \"gram\": %d, \"poly\": %d, \"gemm\": %d}", c ? ", " : "", c,
             P->gram_lists[c].count, P->poly_lists[c].count, P->gemm_lists[c].count);
    j += t;
  }
  j += "], \"launches\": [";
  for (size_t l = 0; l < P->launches.size(); ++l) {
    const Launch& L = P->launches[l];
    snprintf(t, sizeof t, "%s{\"kind\": %d, \"step\": %d, \"chunk\": %d, \"grid\": %d, \"work\": %.17g}",
             l ? ", " : "", L.kind, L.step, L.chunk, L.grid, L.work);
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
  if (P->ptr_event) {
    cudaEventSynchronize(P->ptr_event);
    cudaEventDestroy(P->ptr_event);
  }
  if (P->host_ptrs) cudaFreeHost(P->host_ptrs);
  delete P;
}

}  // extern "C"
