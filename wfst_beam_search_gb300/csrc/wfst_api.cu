// wfst_api.cu — the C ABI (include/wfst_gb300.h): graph upload and
// validation, decoder workspace, offline and streaming calls, lattice export.
//
// Host side of "GPU WFST Beam-Search Decoder" (OASR docs): §4 graph
// validation and the split of the arc columns, §6.1 workspace sizing, §7
// outputs and overflow bits, §8 streaming lifecycle, §10 the C API.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/wfst_gb300.h"
#include "wfst_internal.h"
#include "wfst_vmm.h"

namespace wfst {
cudaError_t launch_decode(const RunArgs& a, int dtype, int grid, cudaStream_t st);
cudaError_t max_grid(int dtype, int L, int* grid);
size_t smem_bytes(int L);
}  // namespace wfst

using namespace wfst;

static thread_local std::string g_err;

static int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}
static int cuda_fail(cudaError_t e, const char* what) {
  return fail(WFST_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CU(call, what)                                   \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
  } while (0)

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

template <typename T>
cudaError_t dev_upload(T** dst, const T* src, size_t n, std::vector<void*>& allocs, int64_t& bytes) {
  *dst = nullptr;
  const size_t b = sizeof(T) * (n ? n : 1);
  cudaError_t e = cudaMalloc((void**)dst, b);
  if (e != cudaSuccess) return e;
  allocs.push_back(*dst);
  bytes += (int64_t)b;
  if (n) e = cudaMemcpy(*dst, src, sizeof(T) * n, cudaMemcpyHostToDevice);
  return e;
}

}  // namespace

struct wfst_graph {
  std::atomic<int> refs{1};
  int device = 0;
  DevGraph dg{};
  std::vector<void*> allocs;
  int64_t bytes = 0;
};

static void graph_release(wfst_graph* g) {
  if (!g) return;
  if (g->refs.fetch_sub(1) == 1) {
    DeviceGuard dgd(g->device);
    for (void* p : g->allocs) cudaFree(p);
    delete g;
  }
}

extern "C" const char* wfst_last_error(void) { return g_err.c_str(); }

extern "C" int wfst_graph_upload(const wfst_graph_desc* d, int32_t device, wfst_graph** out) {
  if (!d || !out) return fail(WFST_ERR_INVALID_ARG, "graph_upload: NULL argument");
  *out = nullptr;
  if (device < 0) return fail(WFST_ERR_INVALID_ARG, "graph_upload: device must be >= 0");
  const int64_t N = d->num_states, A = d->num_arcs, V = d->vocab_size;
  if (N <= 0) return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: num_states must be positive");
  if (A < 0 || A + N >= (int64_t)INT32_MAX)
    return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: num_arcs + num_states must stay below 2^31");
  if (V < 1 || V >= 65535)
    return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: vocab_size must lie in [1, 65535) (u16 ilabels)");
  if (d->start_state < 0 || d->start_state >= N)
    return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: start state out of range");
  if (!d->row_splits || !d->final_weight || (A > 0 && (!d->ilabel || !d->olabel || !d->weight || !d->dst)))
    return fail(WFST_ERR_INVALID_ARG, "graph_upload: NULL array");
  const int64_t* rs = d->row_splits;
  if (rs[0] != 0 || rs[N] != A) return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: row_splits must run 0..num_arcs");
  for (int64_t s = 0; s < N; s++)
    if (rs[s + 1] < rs[s])
      return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: row_splits not monotone at state " + std::to_string(s));
  for (int64_t a = 0; a < A; a++) {
    if (d->dst[a] < 0 || d->dst[a] >= N)
      return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: arc " + std::to_string(a) + " destination out of range");
    if (d->ilabel[a] < -1 || d->ilabel[a] >= V)
      return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: arc " + std::to_string(a) + " ilabel out of range");
    if (std::isnan(d->weight[a]) || d->weight[a] == INFINITY)
      return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: arc " + std::to_string(a) + " weight is NaN or +inf");
  }
  for (int64_t s = 0; s < N; s++)
    if (std::isnan(d->final_weight[s]) || d->final_weight[s] == INFINITY)
      return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: final weight of state " + std::to_string(s) + " is NaN or +inf");

  // epsilon subgraph: acyclic, and its longest path (closure passes needed)
  std::vector<int32_t> indeg(N, 0), depth(N, 0), order;
  bool has_eps = false;
  for (int64_t a = 0; a < A; a++)
    if (d->ilabel[a] < 0) {
      indeg[d->dst[a]]++;
      has_eps = true;
    }
  int32_t eps_depth = 0;
  if (has_eps) {
    order.reserve(N);
    for (int64_t s = 0; s < N; s++)
      if (indeg[s] == 0) order.push_back((int32_t)s);
    for (size_t h = 0; h < order.size(); h++) {
      const int32_t s = order[h];
      for (int64_t a = rs[s]; a < rs[s + 1]; a++)
        if (d->ilabel[a] < 0) {
          const int32_t t = d->dst[a];
          depth[t] = std::max(depth[t], depth[s] + 1);
          eps_depth = std::max(eps_depth, depth[t]);
          if (--indeg[t] == 0) order.push_back(t);
        }
    }
    if ((int64_t)order.size() != N) return fail(WFST_ERR_CORRUPT_GRAPH, "corrupt graph: epsilon arcs form a cycle");
  }

  // internal layout: per state, emitting arcs then epsilon arcs (stable)
  int ndev = 0;
  const cudaError_t ce = cudaGetDeviceCount(&ndev);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(ce, "graph_upload: no CUDA device");
  }
  if (device >= ndev)
    return fail(WFST_ERR_INVALID_ARG, "graph_upload: device " + std::to_string(device) + " is not among the " +
                                          std::to_string(ndev) + " visible CUDA devices");
  std::vector<int4> meta(N);
  std::vector<uint16_t> il16(A ? A : 1);
  std::vector<float> wt(A ? A : 1);
  std::vector<int32_t> dst(A ? A : 1), aid(A ? A : 1), csrc(A ? A : 1);
  for (int64_t s = 0; s < N; s++) {
    int64_t k = rs[s];
    float maxw = -INFINITY;
    for (int pass = 0; pass < 2; pass++) {
      for (int64_t a = rs[s]; a < rs[s + 1]; a++) {
        const bool eps = d->ilabel[a] < 0;
        if (eps != (pass == 1)) continue;
        il16[k] = eps ? (uint16_t)0xFFFF : (uint16_t)d->ilabel[a];
        wt[k] = d->weight[a];
        dst[k] = d->dst[a];
        aid[k] = (int32_t)a;
        if (!eps) maxw = std::max(maxw, d->weight[a]);
        k++;
      }
      if (pass == 0) meta[s].y = (int32_t)k;
    }
    meta[s].x = (int32_t)rs[s];
    meta[s].z = (int32_t)rs[s + 1];
    int32_t bits;
    std::memcpy(&bits, &maxw, 4);
    meta[s].w = bits;
  }
  for (int64_t s = 0; s < N; s++)
    for (int64_t a = rs[s]; a < rs[s + 1]; a++)
      csrc[a] = (int32_t)s | (d->ilabel[a] < 0 ? (int32_t)0x80000000 : 0);

  wfst_graph* g = new wfst_graph();
  g->device = device;
  DeviceGuard dgd(device);
  DevGraph& G = g->dg;
  G.N = (int32_t)N;
  G.start = d->start_state;
  G.V = (int32_t)V;
  G.has_eps = has_eps ? 1 : 0;
  G.A = A;
  G.eps_depth = eps_depth;
  cudaError_t e = cudaSuccess;
  int4* p_meta;
  float* p_fin;
  int32_t *p_csrc, *p_cdst, *p_col;
  if (e == cudaSuccess) e = dev_upload(&p_meta, meta.data(), N, g->allocs, g->bytes);
  if (e == cudaSuccess) e = dev_upload(&p_csrc, csrc.data(), A, g->allocs, g->bytes);
  if (e == cudaSuccess) e = dev_upload(&p_cdst, d->dst, A, g->allocs, g->bytes);
  if (e == cudaSuccess) e = dev_upload(&p_col, d->olabel, A, g->allocs, g->bytes);
  if (e == cudaSuccess) e = dev_upload(&p_fin, d->final_weight, N, g->allocs, g->bytes);
  int4* p_arcs = nullptr;
  if (e == cudaSuccess) {
    std::vector<int4> rec(A ? A : 1);
    for (int64_t k = 0; k < A; k++) {
      int32_t wb;
      std::memcpy(&wb, &wt[k], 4);
      rec[k] = make_int4(dst[k], wb, il16[k] == 0xFFFF ? -1 : (int32_t)il16[k], aid[k]);
    }
    e = dev_upload(&p_arcs, rec.data(), A, g->allocs, g->bytes);
  }
  if (e != cudaSuccess) {
    graph_release(g);
    return e == cudaErrorMemoryAllocation ? fail(WFST_ERR_OOM, "graph_upload: out of device memory")
                                          : cuda_fail(e, "graph_upload");
  }
  G.meta = p_meta;
  G.c_src = p_csrc;
  G.c_dst = p_cdst;
  G.c_olabel = p_col;
  G.final_w = p_fin;
  G.arcs = p_arcs;
  *out = g;
  return WFST_OK;
}

extern "C" int wfst_graph_info(const wfst_graph* g, int64_t* out) {
  if (!g || !out) return fail(WFST_ERR_INVALID_ARG, "graph_info: NULL argument");
  out[0] = g->dg.N;
  out[1] = g->dg.A;
  out[2] = g->dg.V;
  out[3] = g->dg.start;
  out[4] = g->dg.has_eps;
  out[5] = g->dg.eps_depth;
  out[6] = g->bytes;
  out[7] = g->device;
  return WFST_OK;
}

extern "C" void wfst_graph_free(wfst_graph* g) { graph_release(g); }

// Accessors for the other host translation unit (wfst_static.cu).
namespace wfst {
int api_fail(int code, const char* msg) { return fail(code, msg); }
int api_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }
const DevGraph* api_graph(const wfst_graph* g, int* device) {
  *device = g->device;
  return &g->dg;
}
}  // namespace wfst

// ---------------------------------------------------------------------------- decoder

struct wfst_decoder {
  std::mutex mu;
  wfst_graph* g = nullptr;
  wfst_params p{};
  int32_t L = 0, max_frames = 0;
  DevWork w{};
  int grid[2] = {0, 0};
  std::vector<void*> allocs;
  std::vector<size_t> alloc_bytes;
  int64_t bytes = 0;
  int64_t grows = 0;              // capacity doublings so far
  bool path_default = true;       // the best-path buffer has its default size (follows max_frames)
  // pinned host mirrors
  LaneCall* h_calls = nullptr;
  Result* h_res = nullptr;
  LaneState* h_lanes = nullptr;
  LaneStats* h_stats = nullptr;
  GridBar* h_bar = nullptr;
  unsigned long long* h_prof = nullptr;
  int32_t* h_words = nullptr;
  int64_t words_cap_alloc = 0;
  LaneCall* d_calls = nullptr;
  void* d_stage = nullptr;
  size_t stage_bytes = 0;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  // streaming channels
  std::vector<int> chan_state;  // 0 free, 1 open, 2 finalized
  std::vector<int32_t> chan_t;
  std::vector<int> lat_valid;
  int64_t stats[WFST_STAT_COUNT] = {0};
  int64_t test_timeout_ns = 0;    // > 0: the next call's barriers cannot complete (test hook)
  // lazily committed tables (§6.2): worst-case address ranges, physical
  // memory for the current capacities only; growth maps more after it
  LazyRegions lz_front, lz_score, lz_wl;   // [2][L] regions, one stride (entries)
  LazyRegions lz_anc;                      // [2][L], the same stride: ancestor GC (epsilon-free graphs)
  LazyRegions lz_log, lz_bwd;              // [L] regions, one stride
  LazyRegions lz_lat, lz_lat_out;          // [L] regions, one stride
};

// Point the kernel's view at the lazy tables (their bases move when a
// stride grows) and record their strides.
static void sync_lazy(wfst_decoder* d) {
  DevWork& w = d->w;
  w.front = static_cast<TokRec*>(d->lz_front.base());
  w.score = static_cast<float*>(d->lz_score.base());
  w.wl = d->lz_wl.active() ? static_cast<TokRec*>(d->lz_wl.base()) : nullptr;
  w.anc = d->lz_anc.active() ? static_cast<int32_t*>(d->lz_anc.base()) : nullptr;
  w.q_stride = d->lz_front.stride_entries();
  w.wlog = static_cast<int2*>(d->lz_log.base());
  w.bwd = d->lz_bwd.active() ? static_cast<uint32_t*>(d->lz_bwd.base()) : nullptr;
  w.log_stride = d->lz_log.stride_entries();
  w.lat = d->lz_lat.active() ? static_cast<LatRec*>(d->lz_lat.base()) : nullptr;
  w.lat_out = d->lz_lat_out.active() ? static_cast<LatRec*>(d->lz_lat_out.base()) : nullptr;
  w.lat_stride = d->lz_lat.active() ? d->lz_lat.stride_entries() : 0;
}

static int64_t lazy_committed(const wfst_decoder* d) {
  const LazyRegions* r[] = {&d->lz_front, &d->lz_score, &d->lz_wl, &d->lz_anc, &d->lz_log, &d->lz_bwd, &d->lz_lat,
                            &d->lz_lat_out};
  int64_t b = 0;
  for (const LazyRegions* x : r)
    if (x->active()) b += (int64_t)x->committed_bytes();
  return b;
}

static int64_t lazy_reserved(const wfst_decoder* d) {
  const LazyRegions* r[] = {&d->lz_front, &d->lz_score, &d->lz_wl, &d->lz_anc, &d->lz_log, &d->lz_bwd, &d->lz_lat,
                            &d->lz_lat_out};
  int64_t b = 0;
  for (const LazyRegions* x : r)
    if (x->active()) b += (int64_t)x->reserved_bytes();
  return b;
}

// Commit `entries` per region in every active table of a group that shares
// one stride; when that passes the stride, first reserve a common larger
// stride in each of them.  CAPACITY on failure (nothing the call had
// committed is lost).
static int lazy_commit(LazyRegions* const* group, int n, int64_t entries, int64_t floor_stride) {
  std::string msg;
  int64_t stride = 0;
  for (int i = 0; i < n; i++)
    if (group[i]->active()) stride = std::max(stride, group[i]->stride_entries());
  if (entries > stride || floor_stride > stride) {
    const int64_t want = std::max({entries, 2 * stride, floor_stride});
    for (int i = 0; i < n; i++)
      if (group[i]->active() && group[i]->reserve(want, &msg))
        return fail(WFST_ERR_CAPACITY, "lazy tables: " + msg);
    // tables of a group share one stride in entries
    int64_t s = 0;
    for (int i = 0; i < n; i++)
      if (group[i]->active()) s = std::max(s, group[i]->stride_entries());
    for (int i = 0; i < n; i++)
      if (group[i]->active() && group[i]->stride_entries() != s && group[i]->reserve(s, &msg))
        return fail(WFST_ERR_CAPACITY, "lazy tables: " + msg);
  }
  for (int i = 0; i < n; i++)
    if (group[i]->active() && group[i]->commit(entries, &msg)) return fail(WFST_ERR_CAPACITY, "lazy tables: " + msg);
  return WFST_OK;
}

// Winners-log GC: the log of a lane is a ring whose size is a power of two
// (index & (size - 1)) of at most 2^29 entries, so that a signed chain step
// (30 bits) and the two GC marks fit one 32-bit word.
constexpr int64_t kMaxGcRing = (int64_t)1 << 29;
constexpr int64_t kMaxFinCap = (int64_t)1 << 26;  // finalized words per lane
static int64_t gc_ring_size(int64_t want) {
  int64_t r = (int64_t)1 << 10;
  while (r * 2 <= std::min(want, kMaxGcRing)) r *= 2;
  return r;
}

template <typename T>
static cudaError_t dalloc(wfst_decoder* d, T** p, size_t n, bool zero = false) {
  *p = nullptr;
  const size_t b = sizeof(T) * (n ? n : 1);
  cudaError_t e = cudaMalloc((void**)p, b);
  if (e != cudaSuccess) return e;
  d->allocs.push_back(*p);
  d->alloc_bytes.push_back(b);
  d->bytes += (int64_t)b;
  if (zero) e = cudaMemset(*p, 0, b);
  return e;
}

// Swap a workspace array for a freshly allocated one (old contents dropped).
static void dswap(wfst_decoder* d, void** slot, void* fresh, size_t bytes) {
  for (size_t i = 0; i < d->allocs.size(); i++) {
    if (d->allocs[i] != *slot) continue;
    cudaFree(*slot);
    d->bytes -= (int64_t)d->alloc_bytes[i];
    d->allocs.erase(d->allocs.begin() + (long)i);
    d->alloc_bytes.erase(d->alloc_bytes.begin() + (long)i);
    break;
  }
  *slot = fresh;
  d->allocs.push_back(fresh);
  d->alloc_bytes.push_back(bytes);
  d->bytes += (int64_t)bytes;
}

static void decoder_destroy(wfst_decoder* d) {
  if (!d) return;
  {
    DeviceGuard dgd(d->g ? d->g->device : 0);
    cudaDeviceSynchronize();
    d->lz_front.release();
    d->lz_score.release();
    d->lz_wl.release();
    d->lz_anc.release();
    d->lz_log.release();
    d->lz_bwd.release();
    d->lz_lat.release();
    d->lz_lat_out.release();
    for (void* p : d->allocs) cudaFree(p);
    if (d->h_calls) cudaFreeHost(d->h_calls);
    if (d->h_res) cudaFreeHost(d->h_res);
    if (d->h_lanes) cudaFreeHost(d->h_lanes);
    if (d->h_stats) cudaFreeHost(d->h_stats);
    if (d->h_bar) cudaFreeHost(d->h_bar);
    if (d->h_prof) cudaFreeHost(d->h_prof);
    if (d->w.words) cudaFree(d->w.words);
    if (d->h_words) cudaFreeHost(d->h_words);
    if (d->d_stage) cudaFree(d->d_stage);
    if (d->ev0) cudaEventDestroy(d->ev0);
    if (d->ev1) cudaEventDestroy(d->ev1);
  }
  graph_release(d->g);
  delete d;
}

extern "C" int wfst_decoder_create(wfst_graph* g, const wfst_params* params, int32_t max_lanes,
                                   int32_t max_frames, const wfst_capacity* caps, wfst_decoder** out) {
  if (!g || !params || !out) return fail(WFST_ERR_INVALID_ARG, "decoder_create: NULL argument");
  *out = nullptr;
  if (max_lanes < 1 || max_lanes > kMaxLanes)
    return fail(WFST_ERR_INVALID_ARG, "decoder_create: max_lanes must lie in [1, " + std::to_string(kMaxLanes) + "]");
  if (max_frames < 0) return fail(WFST_ERR_INVALID_ARG, "decoder_create: max_frames must be >= 0");
  if (!(params->search_beam > 0.f) || std::isnan(params->output_beam) || params->output_beam < 0.f ||
      params->min_active < 0 || params->max_active < 0)
    return fail(WFST_ERR_INVALID_ARG, "decoder_create: beams must be positive and active bounds >= 0");
  if (params->gc_interval < 0) return fail(WFST_ERR_INVALID_ARG, "decoder_create: gc_interval must be >= 0");
  if (params->lat_prune_interval < 0 || (params->lat_prune_interval > 0 && !params->lattice))
    return fail(WFST_ERR_INVALID_ARG, "decoder_create: lat_prune_interval must be >= 0 and needs lattice = 1");
  if (params->gc_interval > 0 && params->lattice)
    return fail(WFST_ERR_INVALID_ARG,
                "decoder_create: the winners-log GC needs lattice = 0 (lattice records refer to every frame's entries)");
  const bool gc = params->gc_interval > 0;
  const DevGraph& G = g->dg;
  const int64_t N = G.N;
  // lazily committed defaults: the frontier holds up to 16 * max_active
  // tokens (at least 64Ki, at most N) and the winners log 1.5 * max_active
  // entries per frame (at least 1Mi); both grow on overflow
  const int64_t ma = std::max(params->max_active, 1);
  int64_t qcap = (caps && caps->frontier_cap > 0) ? std::min<int64_t>(caps->frontier_cap, N)
                                                  : std::min<int64_t>(N, std::max<int64_t>(65536, 16 * ma));
  const int64_t mf = (int64_t)max_frames + 2;
  int64_t log_cap = (caps && caps->log_cap > 0) ? caps->log_cap : std::max<int64_t>(mf * ma * 3 / 2, 1 << 20);
  log_cap = std::min<int64_t>(log_cap, (int64_t)INT32_MAX - 1);
  if (gc) log_cap = gc_ring_size(log_cap);
  const int64_t fin_cap = gc ? ((caps && caps->fin_cap > 0) ? std::min<int64_t>(caps->fin_cap, kMaxFinCap) : 65536) : 0;
  int64_t lat_cap = 0;
  if (params->lattice)
    lat_cap = (caps && caps->lattice_cap > 0) ? caps->lattice_cap : std::max<int64_t>(mf * ma / 2, 1 << 20);
  // with the GC a backtrack walks only back to the last cut, which can lag
  // the frontier by more than a chunk: room for 4096 frames of arcs
  int64_t path_cap = (caps && caps->path_cap > 0)
                         ? caps->path_cap
                         : 4 * std::max<int64_t>(mf, gc ? 1024 : 0) * (1 + (int64_t)G.eps_depth);
  path_cap = std::min<int64_t>(path_cap, (int64_t)INT32_MAX / 2);
  if (qcap > (int64_t)INT32_MAX || lat_cap > ((int64_t)1 << 40))
    return fail(WFST_ERR_CAPACITY, "decoder_create: capacities exceed the 32-bit tables");

  wfst_decoder* d = new wfst_decoder();
  g->refs.fetch_add(1);
  d->g = g;
  d->p = *params;
  d->L = max_lanes;
  d->max_frames = max_frames;
  d->path_default = !(caps && caps->path_cap > 0);
  DeviceGuard dgd(g->device);
  DevWork& w = d->w;
  w.L = max_lanes;
  w.N = (int32_t)N;
  w.qcap = qcap;
  w.log_cap = log_cap;
  w.log_mask = gc ? (unsigned long long)(log_cap - 1) : ~0ull;
  w.fin_cap = fin_cap;
  w.lat_cap = lat_cap;
  w.path_cap = path_cap;
  w.tiles_cap = G.A / kTile + 2;
  w.lattice = params->lattice ? 1 : 0;
  w.max_frames = max_frames;
  const size_t L = (size_t)max_lanes;
  cudaError_t e = cudaSuccess;
  // the lazy tables: address space for the frontier's worst case (N tokens)
  // and for 8x the initial log and lattice sizes; physical memory for the
  // initial capacities
  const size_t gran = LazyRegions::granularity(g->device);
  if (!gran) {
    decoder_destroy(d);
    return fail(WFST_ERR_CUDA, "decoder_create: CUDA virtual memory management is not available on this device");
  }
  {
    const int64_t q_align = (int64_t)(gran / sizeof(float));       // front, score and worklists share one stride
    const int64_t log_align = (int64_t)(gran / sizeof(uint32_t));  // winners log and bwd share one stride
    const int64_t lat_align = (int64_t)(gran / sizeof(LatRec));
    d->lz_front.init(g->device, 2 * max_lanes, sizeof(TokRec), q_align);
    d->lz_score.init(g->device, 2 * max_lanes, sizeof(float), q_align);
    if (G.has_eps) d->lz_wl.init(g->device, 2 * max_lanes, sizeof(TokRec), q_align);
    if (gc && !G.has_eps) d->lz_anc.init(g->device, 2 * max_lanes, sizeof(int32_t), q_align);
    d->lz_log.init(g->device, max_lanes, sizeof(int2), log_align);
    if (params->lattice) {
      d->lz_bwd.init(g->device, max_lanes, sizeof(uint32_t), log_align);
      d->lz_lat.init(g->device, max_lanes, sizeof(LatRec), lat_align);
      d->lz_lat_out.init(g->device, max_lanes, sizeof(LatRec), lat_align);
    }
    LazyRegions* qg[] = {&d->lz_front, &d->lz_score, &d->lz_wl, &d->lz_anc};
    LazyRegions* lg[] = {&d->lz_log, &d->lz_bwd};
    LazyRegions* ag[] = {&d->lz_lat, &d->lz_lat_out};
    const int64_t log_bound = gc ? kMaxGcRing : (int64_t)INT32_MAX - 1;
    int rc = lazy_commit(qg, 4, qcap, N);
    if (rc == WFST_OK) rc = lazy_commit(lg, 2, log_cap, std::min<int64_t>(8 * log_cap, log_bound));
    if (rc == WFST_OK && params->lattice) rc = lazy_commit(ag, 2, lat_cap, 8 * lat_cap);
    if (rc != WFST_OK) {
      const std::string msg = g_err;
      decoder_destroy(d);
      return fail(WFST_ERR_OOM, "decoder_create: " + msg);
    }
    sync_lazy(d);
  }
#define DA(ptr, n, z) \
  if (e == cudaSuccess) e = dalloc(d, &(ptr), (size_t)(n), z)
  DA(w.ent, 2 * L * N, true);
  if (G.has_eps || params->lattice) DA(w.tpos, L * N, false);  // token positions: epsilon graphs, lattices
  DA(w.maxlp, L * (size_t)std::max(max_frames, 1), false);
  DA(w.tile_first, 2 * L * w.tiles_cap, false);
  if (G.has_eps) {
    DA(w.wl_tile_first, 2 * L * w.tiles_cap, false);
    DA(w.mark, L * N, true);
  }
  DA(w.wl_cnt, 3 * L, true);
  if (gc) DA(w.fin, L * fin_cap, false);
  DA(w.fcnt, 4 * L, true);
  DA(w.lanes, L, true);
  DA(w.stats, L, true);
  if (params->lattice) {
    DA(w.lat_cnt, L, true);
    DA(w.lat_groups, L * (size_t)mf, true);
    DA(w.lat_gtmp, L * (size_t)mf, false);
    DA(w.lat_out_n, L, true);
  }
  DA(w.path, L * path_cap, false);
  DA(w.pframe, L * (size_t)mf, false);
  DA(w.res, L, true);
  DA(w.bar, 1, true);
  DA(w.prof, kProfSlots, true);
  DA(d->d_calls, L, true);
#undef DA
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_calls, sizeof(LaneCall) * L);
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_res, sizeof(Result) * L);
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_lanes, sizeof(LaneState) * L);
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_stats, sizeof(LaneStats) * L);
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_bar, sizeof(GridBar));
  if (e == cudaSuccess) e = cudaMallocHost((void**)&d->h_prof, sizeof(unsigned long long) * kProfSlots);
  if (e == cudaSuccess) e = cudaEventCreate(&d->ev0);
  if (e == cudaSuccess) e = cudaEventCreate(&d->ev1);
  if (e == cudaSuccess) {
    // lanes start free; worklist pass ids start at 1 (marks are 0)
    std::vector<LaneState> init(L);
    for (auto& s : init) {
      std::memset(&s, 0, sizeof(s));
      s.status = kLaneFree;
      s.eps_pass = 1;
      s.t_eff = -1;
    }
    e = cudaMemcpy(w.lanes, init.data(), sizeof(LaneState) * L, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = max_grid(0, max_lanes, &d->grid[0]);
  if (e == cudaSuccess) e = max_grid(1, max_lanes, &d->grid[1]);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    decoder_destroy(d);
    return e == cudaErrorMemoryAllocation
               ? fail(WFST_ERR_OOM, "decoder_create: out of device memory (reduce max_lanes or capacities)")
               : cuda_fail(e, "decoder_create");
  }
  if (d->grid[0] < 1 || d->grid[1] < 1) {
    decoder_destroy(d);
    return fail(WFST_ERR_CUDA, "decoder_create: the decode kernel cannot be made resident");
  }
  d->chan_state.assign(L, 0);
  d->chan_t.assign(L, 0);
  d->lat_valid.assign(L, 0);
  *out = d;
  return WFST_OK;
}

extern "C" void wfst_decoder_free(wfst_decoder* d) { decoder_destroy(d); }

// ---------------------------------------------------------------------------- calls

static int ensure_words(wfst_decoder* d, int32_t words_cap) {
  const int64_t need = (int64_t)d->L * std::max(words_cap, 1);
  if (need <= d->words_cap_alloc) return WFST_OK;
  if (d->w.words) cudaFree(d->w.words);
  if (d->h_words) cudaFreeHost(d->h_words);
  d->w.words = nullptr;
  d->h_words = nullptr;
  d->words_cap_alloc = 0;
  CU(cudaMalloc((void**)&d->w.words, sizeof(int32_t) * need), "words buffer");
  CU(cudaMallocHost((void**)&d->h_words, sizeof(int32_t) * need), "words host buffer");
  d->words_cap_alloc = need;
  return WFST_OK;
}

// Make `lp` device-readable: host input is copied (packed) into a staging buffer.
static int stage_input(wfst_decoder* d, const void* lp, int32_t dtype, int64_t& stride_b, int64_t& stride_t,
                       int32_t B, int32_t T, cudaStream_t st, const void** dev_lp) {
  *dev_lp = lp;
  if (!lp || B == 0 || T == 0) return WFST_OK;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, lp);
  if (e != cudaSuccess) {
    cudaGetLastError();
    at.type = cudaMemoryTypeUnregistered;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    if (at.type == cudaMemoryTypeDevice && at.device != d->g->device)
      return fail(WFST_ERR_INVALID_ARG, "log_probs live on another device than the decoder");
    return WFST_OK;
  }
  const int64_t V = d->g->dg.V;
  const size_t esz = dtype == WFST_F16 ? 2 : 4;
  const size_t need = (size_t)B * T * V * esz;
  if (need > d->stage_bytes) {
    if (d->d_stage) cudaFree(d->d_stage);
    d->d_stage = nullptr;
    d->stage_bytes = 0;
    CU(cudaMalloc(&d->d_stage, need), "host-input staging buffer");
    d->stage_bytes = need;
  }
  const char* src = (const char*)lp;
  char* dst = (char*)d->d_stage;
  if (stride_t == V && stride_b == (int64_t)T * V) {
    CU(cudaMemcpyAsync(dst, src, need, cudaMemcpyHostToDevice, st), "log_probs H2D");
  } else {
    for (int32_t b = 0; b < B; b++)
      CU(cudaMemcpy2DAsync(dst + (size_t)b * T * V * esz, V * esz, src + (size_t)b * stride_b * esz,
                           stride_t * esz, V * esz, T, cudaMemcpyHostToDevice, st),
         "log_probs H2D");
  }
  stride_t = V;
  stride_b = (int64_t)T * V;
  *dev_lp = d->d_stage;
  return WFST_OK;
}

// Run one device call with d->h_calls filled; read back results for lanes in `lanes`.
static int run_call(wfst_decoder* d, const void* lp, int32_t dtype, int64_t stride_b, int64_t stride_t,
                    cudaStream_t st, int32_t words_cap) {
  int rc = ensure_words(d, words_cap);
  if (rc != WFST_OK) return rc;
  const size_t L = (size_t)d->L;
  DevWork& w = d->w;
  CU(cudaMemcpyAsync(d->d_calls, d->h_calls, sizeof(LaneCall) * L, cudaMemcpyHostToDevice, st), "lane calls H2D");
  CU(cudaMemsetAsync(w.bar, 0, sizeof(GridBar), st), "barrier reset");
  CU(cudaMemsetAsync(w.stats, 0, sizeof(LaneStats) * L, st), "stats reset");
  RunArgs a{};
  a.g = d->g->dg;
  a.w = w;
  a.lp = lp;
  a.stride_b = stride_b;
  a.stride_t = stride_t;
  a.calls = d->d_calls;
  a.nlanes = d->L;
  a.words_cap = std::max(words_cap, 1);
  a.search_beam = d->p.search_beam;
  a.output_beam = d->p.output_beam;
  a.min_active = d->p.min_active;
  a.max_active = d->p.max_active;
  a.allow_partial = d->p.allow_partial;
  a.lattice = d->p.lattice;
  a.nblocks = d->grid[dtype == WFST_F16 ? 1 : 0];
  a.ub_skip = (d->p.options & WFST_OPT_NO_UB_SKIP) ? 0 : 1;
  a.gc_interval = d->p.gc_interval;
  a.lat_interval = d->p.lattice ? d->p.lat_prune_interval : 0;
  a.bar_extra = d->test_timeout_ns > 0 ? 1u : 0u;
  a.timeout_ns = d->test_timeout_ns > 0 ? (unsigned long long)d->test_timeout_ns : kBarrierTimeoutNs;
  d->test_timeout_ns = 0;  // one call only
  CU(cudaEventRecord(d->ev0, st), "event");
  CU(launch_decode(a, dtype, a.nblocks, st), "decode kernel launch");
  CU(cudaEventRecord(d->ev1, st), "event");
  CU(cudaMemcpyAsync(d->h_res, w.res, sizeof(Result) * L, cudaMemcpyDeviceToHost, st), "results D2H");
  CU(cudaMemcpyAsync(d->h_lanes, w.lanes, sizeof(LaneState) * L, cudaMemcpyDeviceToHost, st), "lanes D2H");
  CU(cudaMemcpyAsync(d->h_stats, w.stats, sizeof(LaneStats) * L, cudaMemcpyDeviceToHost, st), "stats D2H");
  CU(cudaMemcpyAsync(d->h_bar, w.bar, sizeof(GridBar), cudaMemcpyDeviceToHost, st), "barrier D2H");
  CU(cudaMemcpyAsync(d->h_prof, w.prof, sizeof(unsigned long long) * kProfSlots, cudaMemcpyDeviceToHost, st),
     "phase timers D2H");
  CU(cudaMemcpyAsync(d->h_words, w.words, sizeof(int32_t) * L * a.words_cap, cudaMemcpyDeviceToHost, st),
     "words D2H");
  CU(cudaStreamSynchronize(st), "decode");
  if (d->h_bar->error & 1u) {
    // the call was abandoned mid-way: every lane's state is void (the entry
    // tables and the epsilon dedupe marks, whose pass ids the lanes did not
    // write back, start from zero again)
    cudaMemsetAsync(w.ent, 0, sizeof(ulonglong2) * 2 * L * (size_t)w.N, st);
    if (w.mark) cudaMemsetAsync(w.mark, 0, sizeof(uint32_t) * L * (size_t)w.N, st);
    cudaStreamSynchronize(st);
    for (size_t l = 0; l < L; l++) {
      d->chan_state[l] = 0;
      d->lat_valid[l] = 0;
    }
    return fail(WFST_ERR_TIMEOUT, "decode: a device-side grid barrier wait timed out; the call was abandoned");
  }
  if (d->h_bar->error & 2u) return fail(WFST_ERR_CUDA, "decode: epsilon closure did not converge");
  if (d->h_bar->error & 4u) {
    // a recombination entry kept changing under a bounded CAS loop: the
    // affected lanes' results cannot be trusted; their entries are wiped
    cudaMemsetAsync(d->w.ent, 0, sizeof(ulonglong2) * 2 * L * (size_t)d->w.N, st);
    cudaStreamSynchronize(st);
    for (size_t l = 0; l < L; l++) {
      d->chan_state[l] = 0;
      d->lat_valid[l] = 0;
    }
    return fail(WFST_ERR_TIMEOUT, "decode: a recombination CAS loop gave up after its retry bound");
  }
  float ms = 0.f;
  cudaEventElapsedTime(&ms, d->ev0, d->ev1);
  // per-call counters
  int64_t* S = d->stats;
  std::memset(S, 0, sizeof(d->stats));
  for (size_t l = 0; l < L; l++) {
    if (d->h_calls[l].row < 0) continue;
    const LaneStats& x = d->h_stats[l];
    S[WFST_STAT_FRAMES] += (int64_t)x.frames;
    S[WFST_STAT_SUM_N] += (int64_t)x.sum_n;
    S[WFST_STAT_SUM_D] += (int64_t)x.sum_d;
    S[WFST_STAT_SUM_A] += (int64_t)x.sum_a;
    S[WFST_STAT_SUM_M] += (int64_t)x.sum_m;
    S[WFST_STAT_EPS] += (int64_t)x.eps;
    S[WFST_STAT_ARCS] += (int64_t)(x.sum_d + x.eps + x.finals);
    S[WFST_STAT_STEPS] = std::max<int64_t>(S[WFST_STAT_STEPS], (int64_t)x.steps);
    S[WFST_STAT_LAT_HELD] += (int64_t)x.lat_held;
    S[WFST_STAT_LOG_HW] = std::max<int64_t>(S[WFST_STAT_LOG_HW], (int64_t)x.log_hw);
  }
  S[WFST_STAT_BARRIERS] = d->h_bar->epochs;
  S[WFST_STAT_EPS_PASSES] = d->h_bar->eps_passes;
  S[WFST_STAT_KERNEL_NS] = (int64_t)(ms * 1e6);
  S[WFST_STAT_NS_INIT] = (int64_t)d->h_prof[kProfInit];
  S[WFST_STAT_NS_MAX] = (int64_t)d->h_prof[kProfCommitMax];
  S[WFST_STAT_NS_EXPAND] = (int64_t)d->h_prof[kProfExpand];
  S[WFST_STAT_NS_CLOSURE] = (int64_t)d->h_prof[kProfClosure];
  S[WFST_STAT_NS_PRUNE] = (int64_t)d->h_prof[kProfPrune];
  for (int i = 0; i < 8; i++) S[WFST_STAT_NS_PROLOGUE + i] = (int64_t)d->h_prof[kProfPrologue + i];
  return WFST_OK;
}

// After a call: sanitise lanes whose frontier overflowed (entries that never
// made it into a claims list were not cleared).
static int sanitize(wfst_decoder* d, int32_t lane, cudaStream_t st) {
  const size_t N = (size_t)d->w.N;
  CU(cudaMemsetAsync(d->w.ent + (size_t)lane * N * 2, 0, sizeof(ulonglong2) * 2 * N, st), "sanitise");
  return WFST_OK;
}

static void write_lane(wfst_decoder* d, int32_t lane, int32_t out_index, int32_t* words, int32_t words_cap,
                       int32_t* word_lens, double* scores, int32_t* meta) {
  const Result& r = d->h_res[lane];
  const int ovf = d->h_lanes[lane].overflow;
  const int32_t nw = r.ok ? r.n_words : 0;
  if (words && words_cap > 0) {
    const int32_t k = std::min(nw, words_cap);
    std::memcpy(words + (size_t)out_index * words_cap, d->h_words + (size_t)lane * std::max(words_cap, 1),
                sizeof(int32_t) * k);
  }
  if (word_lens) word_lens[out_index] = nw;
  if (scores) scores[out_index] = r.ok ? (double)r.score : -INFINITY;
  if (meta) {
    meta[3 * out_index + 0] = r.ok;
    meta[3 * out_index + 1] = r.reached_final;
    meta[3 * out_index + 2] = ovf;
  }
}

// Offline capacity growth: double the capacity behind each overflow seen
// (winners log, lattice arena, frontier up to num_states, best path up to the
// longest path a decode can have).  The winners log, lattice arena and
// frontier tables are lazily committed regions: growing them maps more
// physical memory after what each lane holds, so nothing is copied and no
// lane's contents move (only the lanes that overflowed need to run again).
// The best-path and finalized-word buffers are reallocated, every new array
// before any old one is released.  WFST_ERR_CAPACITY when nothing can grow
// (sizes at their bounds, or device memory exhausted): the lanes keep their
// overflow bits.
static int grow_capacities(wfst_decoder* d, bool g_log, bool g_lat, bool g_q, bool g_path) {
  DevWork& w = d->w;
  const size_t L = (size_t)d->L;
  const DevGraph& G = d->g->dg;
  struct Plan { void** slot; size_t bytes; void* fresh; };
  Plan plan[4];
  int np = 0;
  bool grew = false;
  int64_t path_cap = w.path_cap, fin_cap = w.fin_cap;
  const int64_t path_bound = 2 * ((int64_t)d->max_frames + 2) * (1 + (int64_t)G.eps_depth);
  const bool gc = d->p.gc_interval > 0;
  const int64_t log_bound = gc ? kMaxGcRing : (int64_t)INT32_MAX - 1;
  if (g_log && w.log_cap < log_bound) {
    const int64_t cap = std::min<int64_t>(2 * w.log_cap, log_bound);
    LazyRegions* lg[] = {&d->lz_log, &d->lz_bwd};
    if (lazy_commit(lg, 2, cap, 0) != WFST_OK) return WFST_ERR_CAPACITY;
    w.log_cap = cap;
    if (gc) w.log_mask = (unsigned long long)(cap - 1);
    grew = true;
  }
  if (g_lat && w.lattice && w.lat_cap < ((int64_t)1 << 40)) {
    const int64_t cap = 2 * w.lat_cap;
    LazyRegions* ag[] = {&d->lz_lat, &d->lz_lat_out};
    if (lazy_commit(ag, 2, cap, 0) != WFST_OK) return WFST_ERR_CAPACITY;
    w.lat_cap = cap;
    grew = true;
  }
  if (g_q && w.qcap < (int64_t)G.N) {
    const int64_t cap = std::min<int64_t>(2 * w.qcap, (int64_t)G.N);
    LazyRegions* qg[] = {&d->lz_front, &d->lz_score, &d->lz_wl, &d->lz_anc};
    if (lazy_commit(qg, 4, cap, 0) != WFST_OK) return WFST_ERR_CAPACITY;
    w.qcap = cap;
    grew = true;
  }
  sync_lazy(d);
  if (g_path && w.path_cap < path_bound) {
    path_cap = std::min<int64_t>(2 * w.path_cap, path_bound);
    plan[np++] = {(void**)&w.path, sizeof(int32_t) * L * (size_t)path_cap, nullptr};
  }
  if (g_path && gc && w.fin_cap < kMaxFinCap) {  // the finalized-word list shares the path bit
    fin_cap = std::min<int64_t>(2 * w.fin_cap, kMaxFinCap);
    plan[np++] = {(void**)&w.fin, sizeof(int32_t) * L * (size_t)fin_cap, nullptr};
  }
  if (np == 0 && !grew) return fail(WFST_ERR_CAPACITY, "decode: capacities are at their bounds");
  for (int i = 0; i < np; i++) {
    if (cudaMalloc(&plan[i].fresh, plan[i].bytes) != cudaSuccess) {
      cudaGetLastError();
      for (int k = 0; k < i; k++) cudaFree(plan[k].fresh);
      return fail(WFST_ERR_CAPACITY, "decode: no device memory to grow capacities");
    }
  }
  for (int i = 0; i < np; i++) dswap(d, plan[i].slot, plan[i].fresh, plan[i].bytes);
  w.fin_cap = fin_cap;
  w.path_cap = path_cap;
  d->grows++;
  return WFST_OK;
}

// Offline frame-capacity growth (the page's §6 "frame-capacity doubling"):
// an utterance longer than max_frames grows the per-frame tables (row
// maxima, lattice group bounds, per-frame path marks) to max(T, 2 *
// max_frames), and the best-path buffer with them while it has its default
// size.  Every new array is allocated before an old one is released.
static int grow_frames(wfst_decoder* d, int32_t T) {
  DevWork& w = d->w;
  const size_t L = (size_t)d->L;
  const DevGraph& G = d->g->dg;
  const int64_t nf64 = std::max<int64_t>(T, std::min<int64_t>(2 * (int64_t)d->max_frames, (int64_t)INT32_MAX / 8));
  if (nf64 > (int64_t)INT32_MAX / 8) return fail(WFST_ERR_CAPACITY, "decode: T is too large for the frame tables");
  const int32_t nf = (int32_t)nf64;
  const size_t mf = (size_t)nf + 2;
  int64_t path_cap = w.path_cap;
  if (d->path_default) path_cap = std::max<int64_t>(path_cap, 4 * (int64_t)mf * (1 + (int64_t)G.eps_depth));
  struct Plan { void** slot; size_t bytes; void* fresh; bool zero; };
  Plan plan[4];
  int np = 0;
  plan[np++] = {(void**)&w.maxlp, sizeof(float) * L * (size_t)std::max(nf, 1), nullptr, false};
  plan[np++] = {(void**)&w.pframe, sizeof(int2) * L * mf, nullptr, false};
  if (w.lattice) plan[np++] = {(void**)&w.lat_groups, sizeof(int64_t) * L * mf, nullptr, true};
  if (w.lattice) plan[np++] = {(void**)&w.lat_gtmp, sizeof(int64_t) * L * mf, nullptr, false};
  if (path_cap != w.path_cap) plan[np++] = {(void**)&w.path, sizeof(int32_t) * L * (size_t)path_cap, nullptr, false};
  for (int i = 0; i < np; i++) {
    if (cudaMalloc(&plan[i].fresh, plan[i].bytes) != cudaSuccess ||
        (plan[i].zero && cudaMemset(plan[i].fresh, 0, plan[i].bytes) != cudaSuccess)) {
      cudaGetLastError();
      if (plan[i].fresh) cudaFree(plan[i].fresh);
      for (int k = 0; k < i; k++) cudaFree(plan[k].fresh);
      return fail(WFST_ERR_OOM, "decode: no device memory to grow the frame tables");
    }
  }
  for (int i = 0; i < np; i++) dswap(d, plan[i].slot, plan[i].fresh, plan[i].bytes);
  d->max_frames = nf;
  w.max_frames = nf;
  w.path_cap = path_cap;
  return WFST_OK;
}

static void stats_add(int64_t* acc, const int64_t* s) {
  for (int i = 0; i < WFST_STAT_COUNT; i++)
    acc[i] = (i == WFST_STAT_STEPS || i == WFST_STAT_LOG_HW) ? std::max(acc[i], s[i]) : acc[i] + s[i];
}

extern "C" int wfst_decode(wfst_decoder* d, const void* log_probs, int32_t dtype, int64_t stride_b,
                           int64_t stride_t, const int32_t* lens, int32_t B, int32_t T, void* stream,
                           int32_t* words, int32_t words_cap, int32_t* word_lens, double* scores,
                           int32_t* meta) {
  if (!d) return fail(WFST_ERR_INVALID_ARG, "decode: NULL decoder");
  std::lock_guard<std::mutex> lock(d->mu);
  if (d->p.streaming) return fail(WFST_ERR_STATE, "decode: the decoder was created for streaming");
  if (B < 0 || B > d->L) return fail(WFST_ERR_INVALID_ARG, "decode: B must lie in [0, max_lanes]");
  if (T < 0) return fail(WFST_ERR_INVALID_ARG, "decode: T must be >= 0");
  if (T > d->max_frames && (d->p.options & WFST_OPT_NO_GROW))
    return fail(WFST_ERR_INVALID_ARG, "decode: T exceeds max_frames (the decoder was created with WFST_OPT_NO_GROW)");
  if (dtype != WFST_F32 && dtype != WFST_F16) return fail(WFST_ERR_INVALID_ARG, "decode: dtype must be F32 or F16");
  if (words_cap < 0 || (words_cap > 0 && !words)) return fail(WFST_ERR_INVALID_ARG, "decode: bad words buffer");
  if (B == 0) return WFST_OK;
  if (!lens) return fail(WFST_ERR_INVALID_ARG, "decode: NULL lens");
  int32_t maxlen = 0;
  for (int32_t b = 0; b < B; b++) {
    if (lens[b] < 0 || lens[b] > T) return fail(WFST_ERR_INVALID_ARG, "decode: lens[b] must lie in [0, T]");
    maxlen = std::max(maxlen, lens[b]);
  }
  if (maxlen > 0) {
    if (!log_probs) return fail(WFST_ERR_INVALID_ARG, "decode: NULL log_probs");
    if (stride_t < d->g->dg.V || stride_b < 0)
      return fail(WFST_ERR_INVALID_ARG, "decode: stride_t must be >= vocab_size and stride_b >= 0");
  }
  DeviceGuard dgd(d->g->device);
  if (T > d->max_frames) {
    CU(cudaStreamSynchronize((cudaStream_t)stream), "decode: wait before growing the frame tables");
    const int rg = grow_frames(d, T);
    if (rg != WFST_OK) return rg;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const void* lp = log_probs;
  int rc = stage_input(d, log_probs, dtype, stride_b, stride_t, B, T, st, &lp);
  if (rc != WFST_OK) return rc;
  for (int32_t l = 0; l < d->L; l++) {
    LaneCall& c = d->h_calls[l];
    if (l < B) {
      c.row = l;
      c.nframes = lens[l];
      c.flags = kCallInit | kCallFinal;
      c.t_eff = lens[l];
    } else {
      c.row = -1;
      c.nframes = 0;
      c.flags = 0;
      c.t_eff = -1;
    }
  }
  rc = run_call(d, lp, dtype, stride_b, stride_t, st, words_cap);
  if (rc != WFST_OK) return rc;
  int64_t acc[WFST_STAT_COUNT];
  std::memcpy(acc, d->stats, sizeof(acc));
  std::vector<int32_t> ran(B);
  for (int32_t b = 0; b < B; b++) ran[b] = b;
  for (int round = 0;; round++) {
    std::vector<int32_t> over;
    for (int32_t b : ran) {
      write_lane(d, b, b, words, words_cap, word_lens, scores, meta);
      const int ovf = d->h_lanes[b].overflow;
      d->lat_valid[b] = d->p.lattice && d->h_res[b].ok && !(ovf & (kOvfArena | kOvfKept));
      if (ovf & kOvfKept) {
        rc = sanitize(d, b, st);
        if (rc != WFST_OK) return rc;
      }
      if (ovf & (kOvfArena | kOvfKept | kOvfPath)) over.push_back(b);
    }
    if (over.empty() || (d->p.options & WFST_OPT_NO_GROW) || round >= kMaxGrowRounds) break;
    bool g_log = false, g_lat = false, g_q = false, g_path = false;
    std::vector<unsigned long long> lat_n;
    if (d->p.lattice) {
      lat_n.resize(d->L);
      CU(cudaMemcpyAsync(lat_n.data(), d->w.lat_cnt, sizeof(unsigned long long) * d->L, cudaMemcpyDeviceToHost, st),
         "lattice counts D2H");
      CU(cudaStreamSynchronize(st), "lattice counts D2H");
    }
    for (int32_t b : over) {
      const int ovf = d->h_lanes[b].overflow;
      if (ovf & kOvfKept) g_q = true;
      if (ovf & kOvfPath) g_path = true;
      if (ovf & kOvfArena) {
        const bool lat_full = d->p.lattice && lat_n[b] > (unsigned long long)d->w.lat_cap;
        if (lat_full) g_lat = true;
        if (d->h_lanes[b].cursor > d->w.log_cap || !lat_full) g_log = true;
      }
    }
    rc = grow_capacities(d, g_log, g_lat, g_q, g_path);
    if (rc == WFST_ERR_CAPACITY) break;  // already at the largest sizes: the bits stay set
    if (rc != WFST_OK) return rc;
    // the grown tables kept every lane's contents in place: only the lanes
    // that overflowed run again
    ran = over;
    for (int32_t l = 0; l < d->L; l++) d->h_calls[l].row = -1;
    for (int32_t b : ran) {
      LaneCall& c = d->h_calls[b];
      c.row = b;
      c.nframes = lens[b];
      c.flags = kCallInit | kCallFinal;
      c.t_eff = lens[b];
    }
    rc = run_call(d, lp, dtype, stride_b, stride_t, st, words_cap);
    if (rc != WFST_OK) return rc;
    stats_add(acc, d->stats);
  }
  std::memcpy(d->stats, acc, sizeof(acc));
  if (d->p.lattice) {  // records held after the last round (a re-run replaced a lane's records)
    std::vector<unsigned long long> held(B);
    CU(cudaMemcpyAsync(held.data(), d->w.lat_cnt, sizeof(unsigned long long) * B, cudaMemcpyDeviceToHost, st),
       "lattice counts D2H");
    CU(cudaStreamSynchronize(st), "lattice counts D2H");
    d->stats[WFST_STAT_LAT_HELD] = 0;
    for (int32_t b = 0; b < B; b++)
      d->stats[WFST_STAT_LAT_HELD] += (int64_t)std::min<unsigned long long>(held[b], (unsigned long long)d->w.lat_cap);
  }
  CU(cudaStreamSynchronize(st), "decode");
  return WFST_OK;
}

// Streaming headroom: a channel cannot grow a table in the middle of a call,
// but between calls the lazily committed winners log and lattice arena grow
// in place (their contents stay where they are), so when an open channel
// has used more than half of either, double it: a stream then overflows
// only if one chunk adds more than half a table.  Not for the winners-log
// GC's rings, whose index mask depends on their size.
static int stream_headroom(wfst_decoder* d, cudaStream_t st) {
  DevWork& w = d->w;
  int64_t log_use = 0, lat_use = 0;
  for (int32_t l = 0; l < d->L; l++)
    if (d->chan_state[l] == 1) log_use = std::max<int64_t>(log_use, d->h_lanes[l].cursor - d->h_lanes[l].floor);
  if (d->p.lattice) {
    std::vector<unsigned long long> n(d->L);
    CU(cudaMemcpyAsync(n.data(), w.lat_cnt, sizeof(unsigned long long) * d->L, cudaMemcpyDeviceToHost, st),
       "lattice counts D2H");
    CU(cudaStreamSynchronize(st), "lattice counts D2H");
    for (int32_t l = 0; l < d->L; l++)
      if (d->chan_state[l] == 1) lat_use = std::max<int64_t>(lat_use, (int64_t)n[l]);
  }
  const bool g_log = d->p.gc_interval == 0 && log_use > w.log_cap / 2 && w.log_cap < (int64_t)INT32_MAX / 2;
  const bool g_lat = d->p.lattice && lat_use > w.lat_cap / 2;
  if (!g_log && !g_lat) return WFST_OK;
  CU(cudaStreamSynchronize(st), "stream headroom");
  const int rc = grow_capacities(d, g_log, g_lat, false, false);
  return rc == WFST_ERR_CAPACITY ? WFST_OK : rc;  // no room: the channels keep running until they overflow
}

static bool rec_less(const wfst_lat_record& x, const wfst_lat_record& y) {
  if (x.t != y.t) return x.t < y.t;
  if (x.src_state != y.src_state) return x.src_state < y.src_state;
  return x.arc_id < y.arc_id;
}

extern "C" int wfst_lattice_export(wfst_decoder* d, int32_t lane, wfst_lat_record* out, int64_t cap,
                                   int64_t* n_records) {
  if (!d || !n_records) return fail(WFST_ERR_INVALID_ARG, "lattice_export: NULL argument");
  std::lock_guard<std::mutex> lock(d->mu);
  if (!d->p.lattice) return fail(WFST_ERR_STATE, "lattice_export: the decoder was created without lattice");
  if (lane < 0 || lane >= d->L) return fail(WFST_ERR_INVALID_ARG, "lattice_export: lane out of range");
  *n_records = 0;
  if (!d->lat_valid[lane]) return WFST_OK;
  DeviceGuard dgd(d->g->device);
  unsigned long long n = 0;
  CU(cudaMemcpy(&n, d->w.lat_out_n + lane, sizeof(n), cudaMemcpyDeviceToHost), "lattice count");
  n = std::min<unsigned long long>(n, (unsigned long long)d->w.lat_cap);
  std::vector<LatRec> recs(n);
  if (n)
    CU(cudaMemcpy(recs.data(), d->w.lat_out + (size_t)lane * d->w.lat_stride, sizeof(LatRec) * n,
                  cudaMemcpyDeviceToHost),
       "lattice D2H");
  std::vector<wfst_lat_record> o(n);
  for (size_t i = 0; i < n; i++) {
    const LatRec& r = recs[i];
    o[i].t = r.frame_flags >> 4;
    o[i].src_state = r.src_state;
    o[i].dst_state = r.dst_state;
    o[i].arc_id = r.arc;
    o[i].flags = r.frame_flags & (kRecEps | kRecFinal | kRecRedirect);
    o[i].score = r.arcscore;
  }
  std::sort(o.begin(), o.end(), rec_less);
  // One record per (source token, arc): an epsilon arc of a token whose key
  // changed during the closure without changing its score (a tie won by a
  // lower arc id, or an improvement that landed before the token's own tile
  // staged it) is relaxed in two passes with the same final score.  Both
  // relaxations pass the device's final-score check and are identical.
  size_t k = 0;
  for (size_t i = 0; i < o.size(); i++)
    if (k == 0 || rec_less(o[k - 1], o[i])) o[k++] = o[i];
  o.resize(k);
  *n_records = (int64_t)k;
  if (out && cap > 0) std::memcpy(out, o.data(), sizeof(wfst_lat_record) * std::min<int64_t>(cap, (int64_t)k));
  return WFST_OK;
}

// ---------------------------------------------------------------------------- streaming

static void calls_idle(wfst_decoder* d) {
  for (int32_t l = 0; l < d->L; l++) {
    d->h_calls[l].row = -1;
    d->h_calls[l].nframes = 0;
    d->h_calls[l].flags = 0;
    d->h_calls[l].t_eff = -1;
  }
}

extern "C" int wfst_stream_create(wfst_decoder* d, int32_t* channel) {
  if (!d || !channel) return fail(WFST_ERR_INVALID_ARG, "stream_create: NULL argument");
  std::lock_guard<std::mutex> lock(d->mu);
  if (!d->p.streaming) return fail(WFST_ERR_STATE, "stream_create: the decoder was created for offline decoding");
  *channel = -1;
  int32_t ch = -1;
  for (int32_t l = 0; l < d->L; l++)
    if (d->chan_state[l] == 0) {
      ch = l;
      break;
    }
  if (ch < 0) return WFST_OK;
  DeviceGuard dgd(d->g->device);
  calls_idle(d);
  d->h_calls[ch] = LaneCall{0, 0, kCallInit, -1};
  int rc = run_call(d, nullptr, WFST_F32, 0, 0, (cudaStream_t)0, 1);
  if (rc != WFST_OK) return rc;
  d->chan_state[ch] = 1;
  d->chan_t[ch] = 0;
  d->lat_valid[ch] = 0;
  *channel = ch;
  return WFST_OK;
}

static int check_channels(wfst_decoder* d, const int32_t* channels, int32_t n, int want_state) {
  if (n < 0 || n > d->L || (n > 0 && !channels)) return fail(WFST_ERR_INVALID_ARG, "bad channel list");
  std::vector<int> seen(d->L, 0);
  for (int32_t i = 0; i < n; i++) {
    const int32_t c = channels[i];
    if (c < 0 || c >= d->L) return fail(WFST_ERR_INVALID_ARG, "channel id out of range");
    if (seen[c]++) return fail(WFST_ERR_INVALID_ARG, "channel listed twice");
    if (d->chan_state[c] != want_state) return fail(WFST_ERR_STATE, "channel " + std::to_string(c) + " is not open");
  }
  return WFST_OK;
}

extern "C" int wfst_stream_advance(wfst_decoder* d, const int32_t* channels, int32_t n, const void* log_probs,
                                   int32_t dtype, int64_t stride_b, int64_t stride_t, const int32_t* chunk_lens,
                                   int32_t chunk_T, int32_t want_partial, void* stream, int32_t* words,
                                   int32_t words_cap, int32_t* word_lens, double* scores, int32_t* meta) {
  if (!d) return fail(WFST_ERR_INVALID_ARG, "stream_advance: NULL decoder");
  std::lock_guard<std::mutex> lock(d->mu);
  if (!d->p.streaming) return fail(WFST_ERR_STATE, "stream_advance: not a streaming decoder");
  int rc = check_channels(d, channels, n, 1);
  if (rc != WFST_OK) return rc;
  if (dtype != WFST_F32 && dtype != WFST_F16) return fail(WFST_ERR_INVALID_ARG, "stream_advance: bad dtype");
  if (chunk_T < 0 || (n > 0 && !chunk_lens)) return fail(WFST_ERR_INVALID_ARG, "stream_advance: bad chunk lengths");
  if (chunk_T > d->max_frames)
    return fail(WFST_ERR_INVALID_ARG, "stream_advance: chunk_T must not exceed the decoder's max_frames");
  int32_t maxlen = 0;
  for (int32_t i = 0; i < n; i++) {
    if (chunk_lens[i] < 0 || chunk_lens[i] > chunk_T)
      return fail(WFST_ERR_INVALID_ARG, "stream_advance: chunk_lens[i] must lie in [0, chunk_T]");
    if (d->p.lattice && d->chan_t[channels[i]] + chunk_lens[i] > d->max_frames)
      return fail(WFST_ERR_INVALID_ARG, "stream_advance: a lattice stream cannot exceed max_frames");
    maxlen = std::max(maxlen, chunk_lens[i]);
  }
  if (maxlen > 0 && (!log_probs || stride_t < d->g->dg.V || stride_b < 0))
    return fail(WFST_ERR_INVALID_ARG, "stream_advance: bad log_probs or strides");
  if (want_partial && words_cap < 0) return fail(WFST_ERR_INVALID_ARG, "stream_advance: bad words_cap");
  if (n == 0) return WFST_OK;
  DeviceGuard dgd(d->g->device);
  cudaStream_t st = (cudaStream_t)stream;
  const void* lp = log_probs;
  rc = stage_input(d, log_probs, dtype, stride_b, stride_t, n, chunk_T, st, &lp);
  if (rc != WFST_OK) return rc;
  calls_idle(d);
  for (int32_t i = 0; i < n; i++)
    d->h_calls[channels[i]] = LaneCall{i, chunk_lens[i], want_partial ? kCallPartial : 0, -1};
  rc = run_call(d, lp, dtype, stride_b, stride_t, st, want_partial ? words_cap : 1);
  if (rc != WFST_OK) return rc;
  rc = stream_headroom(d, st);
  if (rc != WFST_OK) return rc;
  for (int32_t i = 0; i < n; i++) {
    d->chan_t[channels[i]] += chunk_lens[i];
    if (want_partial) {
      write_lane(d, channels[i], i, words, words_cap, word_lens, scores, meta);
      if (meta) meta[3 * i + 1] = 0;
    }
  }
  return WFST_OK;
}

extern "C" int wfst_stream_finalize(wfst_decoder* d, const int32_t* channels, int32_t n, void* stream,
                                    int32_t* words, int32_t words_cap, int32_t* word_lens, double* scores,
                                    int32_t* meta) {
  if (!d) return fail(WFST_ERR_INVALID_ARG, "stream_finalize: NULL decoder");
  std::lock_guard<std::mutex> lock(d->mu);
  if (!d->p.streaming) return fail(WFST_ERR_STATE, "stream_finalize: not a streaming decoder");
  int rc = check_channels(d, channels, n, 1);
  if (rc != WFST_OK) return rc;
  if (words_cap < 0 || (words_cap > 0 && !words)) return fail(WFST_ERR_INVALID_ARG, "stream_finalize: bad words buffer");
  if (n == 0) return WFST_OK;
  DeviceGuard dgd(d->g->device);
  cudaStream_t st = (cudaStream_t)stream;
  calls_idle(d);
  for (int32_t i = 0; i < n; i++) d->h_calls[channels[i]] = LaneCall{0, 0, kCallFinal, -1};
  rc = run_call(d, nullptr, WFST_F32, 0, 0, st, words_cap);
  if (rc != WFST_OK) return rc;
  for (int32_t i = 0; i < n; i++) {
    const int32_t c = channels[i];
    write_lane(d, c, i, words, words_cap, word_lens, scores, meta);
    const int ovf = d->h_lanes[c].overflow;
    d->lat_valid[c] = d->p.lattice && d->h_res[c].ok && !(ovf & (kOvfArena | kOvfKept));
    d->chan_state[c] = 2;
  }
  return WFST_OK;
}

extern "C" int wfst_stream_release(wfst_decoder* d, int32_t channel) {
  if (!d) return fail(WFST_ERR_INVALID_ARG, "stream_release: NULL decoder");
  std::lock_guard<std::mutex> lock(d->mu);
  if (channel < 0 || channel >= d->L || d->chan_state[channel] == 0)
    return fail(WFST_ERR_INVALID_ARG, "stream_release: channel is not in use");
  DeviceGuard dgd(d->g->device);
  // a finalized channel's entries were cleared by its final step, unless
  // tokens were dropped past the frontier capacity
  if (d->chan_state[channel] != 2 || (d->h_lanes[channel].overflow & kOvfKept)) {
    int rc = sanitize(d, channel, (cudaStream_t)0);
    if (rc != WFST_OK) return rc;
  }
  LaneState s;
  std::memset(&s, 0, sizeof(s));
  CU(cudaMemcpy(&s.eps_pass, &d->w.lanes[channel].eps_pass, sizeof(uint32_t), cudaMemcpyDeviceToHost), "release");
  s.status = kLaneFree;
  s.t_eff = -1;
  CU(cudaMemcpy(d->w.lanes + channel, &s, sizeof(s), cudaMemcpyHostToDevice), "release");
  d->chan_state[channel] = 0;
  d->chan_t[channel] = 0;
  d->lat_valid[channel] = 0;
  return WFST_OK;
}

extern "C" int wfst_test_barrier_timeout(wfst_decoder* d, int64_t timeout_ns) {
  if (!d) return fail(WFST_ERR_INVALID_ARG, "test_barrier_timeout: NULL decoder");
  if (timeout_ns < 1000000 || timeout_ns > (int64_t)kBarrierTimeoutNs)
    return fail(WFST_ERR_INVALID_ARG, "test_barrier_timeout: timeout_ns must lie in [1 ms, 4 s]");
  std::lock_guard<std::mutex> lock(d->mu);
  d->test_timeout_ns = timeout_ns;
  return WFST_OK;
}

extern "C" int wfst_mem_stats(wfst_decoder* d, int64_t* out, int32_t n) {
  if (!d || !out || n < 0) return fail(WFST_ERR_INVALID_ARG, "mem_stats: bad argument");
  std::lock_guard<std::mutex> lock(d->mu);
  const int64_t lazy = lazy_committed(d);
  const int64_t v[WFST_MEM_COUNT] = {d->bytes + lazy, d->w.qcap, d->w.log_cap, d->w.lat_cap, d->w.path_cap, d->grows,
                                     d->max_frames, lazy_reserved(d), lazy};
  for (int32_t i = 0; i < n && i < WFST_MEM_COUNT; i++) out[i] = v[i];
  return WFST_OK;
}

extern "C" int wfst_stats(wfst_decoder* d, int64_t* out, int32_t n) {
  if (!d || !out || n < 0) return fail(WFST_ERR_INVALID_ARG, "stats: bad argument");
  std::lock_guard<std::mutex> lock(d->mu);
  for (int32_t i = 0; i < n && i < WFST_STAT_COUNT; i++) out[i] = d->stats[i];
  return WFST_OK;
}
