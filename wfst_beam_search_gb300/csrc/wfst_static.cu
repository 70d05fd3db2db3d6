// wfst_static.cu — wfst_decode_static: an offline decode whose working memory
// is one fixed region of device memory that the library declares statically,
// so that the call itself allocates nothing (no cudaMalloc/cudaFree, no pinned
// host buffers, no allocating library routine).
//
// Who needs it: callers that must not allocate device memory once they run —
// a process whose memory is handed out by its own pool and may not grow
// behind that pool's back, a real-time audio thread that must not block in
// the allocator, or an embedding that sizes device memory once at start-up.
// The web page "GPU WFST Beam-Search Decoder" has no counterpart for this
// entry point; it runs the same decode kernel as wfst_decode.
//
// The region is file-scope `__device__` storage of kScratchBytes.  Its
// address is taken once per device (with that device current) through
// cudaGetSymbolAddress; that first lookup may load the module onto the
// device, so make the first call before any stream capture begins.
//
// Limits: B <= kStaticLanes lanes, lattice and streaming off, and the call's
// fixed tables (sized from B, T, the graph and words_cap) must fit the region;
// a call that does not fit returns WFST_ERR_CAPACITY with the bytes it
// needed.  The winners log gets the rest of the region, up to the most a
// call can use (one entry per state and frame).  It cannot grow: a lane that
// fills it comes back with overflow bit 4, and the call then returns
// WFST_ERR_CAPACITY (the outputs are still written, flagged), where
// wfst_decode would grow the log and decode the lane again.
//
// Zeroing: the recombination entries, the epsilon dedupe marks, the frame and
// worklist counters, the grid barrier, the statistics and the result slots
// must start at zero.  They sit at the front of the layout and every call
// clears that front part with cudaMemsetAsync before its launch; everything
// after it is written before it is read.
//
// Concurrency: the region is one per device per process.  Two calls on the
// same device that overlapped would race on it, so the call holds a
// per-device lock from its first write of the region until its stream work
// has finished — on every return path, errors included.  Separate processes
// each have their own region.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/wfst_gb300.h"
#include "wfst_internal.h"

namespace wfst {
cudaError_t launch_decode(const RunArgs& a, int dtype, int grid, cudaStream_t st);
cudaError_t max_grid(int dtype, int L, int* grid);
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
const DevGraph* api_graph(const wfst_graph* g, int* device);
}  // namespace wfst

using namespace wfst;

namespace {

constexpr size_t kScratchBytes = (size_t)WFST_STATIC_SCRATCH_BYTES;
constexpr int kStaticLanes = WFST_STATIC_MAX_LANES;
constexpr int kMaxDevices = 64;

static_assert(kStaticLanes <= kMaxLanes, "static lanes exceed the kernel's lane table");

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSlot {
  std::mutex mu;            // held for a whole call: the region is shared by all calls on the device
  bool ready = false;
  unsigned char* base = nullptr;
  int grid[2] = {0, 0};
};
DeviceSlot g_slots[kMaxDevices];

struct Lens {
  int32_t v[kStaticLanes];
};

// Lane states and per-call lane records of a fresh offline call: every lane
// starts free with worklist pass id 1 (the marks were just zeroed).
__global__ void static_prepare(LaneState* lanes, LaneCall* calls, Lens lens, int B) {
  const int l = threadIdx.x;
  if (l >= B) return;
  LaneState s;
  memset(&s, 0, sizeof(s));
  s.status = kLaneFree;
  s.eps_pass = 1;
  s.t_eff = -1;
  lanes[l] = s;
  LaneCall c;
  c.row = l;
  c.nframes = lens.v[l];
  c.flags = kCallInit | kCallFinal;
  c.t_eff = lens.v[l];
  calls[l] = c;
}

// Bump allocator over the region: 256-byte aligned sub-arrays.
struct Carve {
  unsigned char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += sizeof(T) * (n ? n : 1);
    return p;
  }
};

// Lays the call's tables out from `base` (nullptr: size only) with a winners
// log of `log_cap` entries per lane.  Returns the total bytes and, in
// *zero_bytes, the length of the front part that must start at zero.
size_t layout(unsigned char* base, const DevGraph& G, int L, int T, int64_t log_cap, int words_cap,
              DevWork& w, LaneCall** calls, size_t* zero_bytes) {
  Carve c{base};
  const size_t N = (size_t)G.N;
  const int64_t mf = (int64_t)T + 2;
  w = DevWork{};
  w.L = L;
  w.N = G.N;
  w.qcap = G.N;
  w.log_cap = log_cap;
  w.log_mask = ~0ull;  // a flat log (no winners-log GC here)
  w.lat_cap = 0;
  w.q_stride = w.qcap;  // flat tables: one lane's region after another
  w.log_stride = w.log_cap;
  w.lat_stride = 0;
  w.path_cap = 4 * mf * (1 + (int64_t)G.eps_depth);
  w.tiles_cap = G.A / kTile + 2;
  w.lattice = 0;
  w.max_frames = T;
  // the front part: everything that must start at zero
  w.bar = c.take<GridBar>(1);
  w.prof = c.take<unsigned long long>(kProfSlots);
  w.stats = c.take<LaneStats>(L);
  w.res = c.take<Result>(L);
  w.fcnt = c.take<FrameCnt>(4 * (size_t)L);
  w.wl_cnt = c.take<unsigned long long>(3 * (size_t)L);
  w.ent = c.take<ulonglong2>(2 * (size_t)L * N);
  if (G.has_eps) w.mark = c.take<uint32_t>((size_t)L * N);
  *zero_bytes = (c.off + 255) & ~(size_t)255;
  // the rest: written before it is read
  w.lanes = c.take<LaneState>(L);
  *calls = c.take<LaneCall>(L);
  w.tpos = c.take<int2>((size_t)L * N);
  w.front = c.take<TokRec>(2 * (size_t)L * w.qcap);
  w.score = c.take<float>(2 * (size_t)L * w.qcap);
  w.maxlp = c.take<float>((size_t)L * std::max(T, 1));
  w.tile_first = c.take<int32_t>(2 * (size_t)L * w.tiles_cap);
  if (G.has_eps) {
    w.wl = c.take<TokRec>(2 * (size_t)L * w.qcap);
    w.wl_tile_first = c.take<int32_t>(2 * (size_t)L * w.tiles_cap);
  }
  w.path = c.take<int32_t>((size_t)L * w.path_cap);
  w.pframe = c.take<int2>((size_t)L * mf);
  w.words = c.take<int32_t>((size_t)L * words_cap);
  w.wlog = c.take<int2>((size_t)L * w.log_cap);  // last: it takes what is left
  return (c.off + 255) & ~(size_t)255;
}

// First use on a device (that device current): resolve the region's address
// and the cooperative grid of both input types.
int setup_device(DeviceSlot& s) {
  if (s.ready) return WFST_OK;
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
  if (e != cudaSuccess) return api_cuda_fail(e, "decode_static: cudaGetSymbolAddress of the scratch region");
  if (!ptr) return api_fail(WFST_ERR_CUDA, "decode_static: the scratch region has no device address");
  e = max_grid(0, kStaticLanes, &s.grid[0]);
  if (e == cudaSuccess) e = max_grid(1, kStaticLanes, &s.grid[1]);
  if (e != cudaSuccess) return api_cuda_fail(e, "decode_static: occupancy query");
  if (s.grid[0] < 1 || s.grid[1] < 1)
    return api_fail(WFST_ERR_CUDA, "decode_static: the decode kernel cannot be made resident");
  s.base = static_cast<unsigned char*>(ptr);
  s.ready = true;
  return WFST_OK;
}

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

#define CUS(call, what)                                  \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return api_cuda_fail(e_, what); \
  } while (0)

// Waits for the call's stream work on every return once armed, so that the
// per-device lock (released after this guard) is never given up while a
// kernel or a copy of this call still uses the region.
struct StreamDrain {
  cudaStream_t st;
  bool armed = false;
  ~StreamDrain() {
    if (armed) cudaStreamSynchronize(st);
  }
};

}  // namespace

extern "C" int wfst_decode_static(const wfst_graph* g, const wfst_params* params, const void* log_probs,
                                  int32_t dtype, int64_t stride_b, int64_t stride_t, const int32_t* lens,
                                  int32_t B, int32_t T, void* stream, int32_t* words, int32_t words_cap,
                                  int32_t* word_lens, double* scores, int32_t* meta) {
  if (!g || !params) return api_fail(WFST_ERR_INVALID_ARG, "decode_static: NULL graph or params");
  if (params->lattice || params->streaming || params->gc_interval || params->lat_prune_interval)
    return api_fail(WFST_ERR_INVALID_ARG,
                    "decode_static: lattice, streaming, gc_interval and lat_prune_interval must be 0");
  if (!(params->search_beam > 0.f) || std::isnan(params->output_beam) || params->output_beam < 0.f ||
      params->min_active < 0 || params->max_active < 0)
    return api_fail(WFST_ERR_INVALID_ARG, "decode_static: beams must be positive and active bounds >= 0");
  if (B < 0 || B > kStaticLanes)
    return api_fail(WFST_ERR_CAPACITY, "decode_static: B exceeds WFST_STATIC_MAX_LANES (8)");
  if (T < 0) return api_fail(WFST_ERR_INVALID_ARG, "decode_static: T must be >= 0");
  if (dtype != WFST_F32 && dtype != WFST_F16)
    return api_fail(WFST_ERR_INVALID_ARG, "decode_static: dtype must be F32 or F16");
  if (words_cap < 0 || (words_cap > 0 && !words))
    return api_fail(WFST_ERR_INVALID_ARG, "decode_static: bad words buffer");
  if (B == 0) return WFST_OK;
  if (!lens) return api_fail(WFST_ERR_INVALID_ARG, "decode_static: NULL lens");
  Lens lv{};
  int32_t maxlen = 0;
  for (int32_t b = 0; b < B; b++) {
    if (lens[b] < 0 || lens[b] > T) return api_fail(WFST_ERR_INVALID_ARG, "decode_static: lens[b] must lie in [0, T]");
    lv.v[b] = lens[b];
    maxlen = std::max(maxlen, lens[b]);
  }
  int device = 0;
  const DevGraph* G = api_graph(g, &device);
  if (device < 0 || device >= kMaxDevices)
    return api_fail(WFST_ERR_INVALID_ARG, "decode_static: device index beyond the supported range");
  if (maxlen > 0) {
    if (!log_probs) return api_fail(WFST_ERR_INVALID_ARG, "decode_static: NULL log_probs");
    if (stride_t < G->V || stride_b < 0)
      return api_fail(WFST_ERR_INVALID_ARG, "decode_static: stride_t must be >= vocab_size and stride_b >= 0");
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, log_probs);
    if (e != cudaSuccess) {
      cudaGetLastError();
      at.type = cudaMemoryTypeUnregistered;
    }
    if (!((at.type == cudaMemoryTypeDevice && at.device == device) || at.type == cudaMemoryTypeManaged))
      return api_fail(WFST_ERR_INVALID_ARG, "decode_static: log_probs must be device memory on the graph's device");
  }
  const int wc = std::max(words_cap, 1);
  DevWork w;
  LaneCall* calls = nullptr;
  size_t zero_bytes = 0;
  // the fixed tables with a log of one entry per frame, then the log takes
  // the rest of the region up to one entry per state and frame
  const int64_t mf = (int64_t)T + 2;
  const size_t fixed = layout(nullptr, *G, B, T, mf, wc, w, &calls, &zero_bytes);
  if (fixed > kScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "decode_static: the call needs %zu bytes of scratch, above WFST_STATIC_SCRATCH_BYTES (%zu)",
             fixed, kScratchBytes);
    return api_fail(WFST_ERR_CAPACITY, msg);
  }
  const int64_t log_bound = mf * (int64_t)G->N;
  const int64_t log_room = mf + (int64_t)((kScratchBytes - fixed) / (sizeof(int2) * (size_t)B));
  const int64_t log_cap = std::min<int64_t>(std::min(log_bound, log_room), (int64_t)INT32_MAX - 1);

  DeviceSlot& slot = g_slots[device];
  std::lock_guard<std::mutex> lock(slot.mu);
  DeviceGuard dgd(device);
  int rc = setup_device(slot);
  if (rc != WFST_OK) return rc;
  const size_t used = layout(slot.base, *G, B, T, log_cap, wc, w, &calls, &zero_bytes);
  if (used > kScratchBytes) return api_fail(WFST_ERR_CAPACITY, "decode_static: internal layout error");
  cudaStream_t st = (cudaStream_t)stream;
  StreamDrain drain{st};  // destroyed before `lock`: the stream is drained first
  drain.armed = true;
  CUS(cudaMemsetAsync(slot.base, 0, zero_bytes, st), "decode_static: scratch clear");
  static_prepare<<<1, 32, 0, st>>>(w.lanes, calls, lv, B);
  CUS(cudaGetLastError(), "decode_static: lane set-up launch");
  RunArgs a{};
  a.g = *G;
  a.w = w;
  a.lp = log_probs;
  a.stride_b = stride_b;
  a.stride_t = stride_t;
  a.calls = calls;
  a.nlanes = B;
  a.words_cap = wc;
  a.search_beam = params->search_beam;
  a.output_beam = params->output_beam;
  a.min_active = params->min_active;
  a.max_active = params->max_active;
  a.allow_partial = params->allow_partial;
  a.lattice = 0;
  a.nblocks = slot.grid[dtype == WFST_F16 ? 1 : 0];
  a.ub_skip = (params->options & WFST_OPT_NO_UB_SKIP) ? 0 : 1;
  a.timeout_ns = kBarrierTimeoutNs;
  CUS(launch_decode(a, dtype, a.nblocks, st), "decode_static: decode kernel launch");
  // results into host stack memory (pageable copies; the call then waits)
  Result res[kStaticLanes];
  LaneState lanes[kStaticLanes];
  GridBar bar;
  CUS(cudaMemcpyAsync(res, w.res, sizeof(Result) * B, cudaMemcpyDeviceToHost, st), "decode_static: results D2H");
  CUS(cudaMemcpyAsync(lanes, w.lanes, sizeof(LaneState) * B, cudaMemcpyDeviceToHost, st),
      "decode_static: lanes D2H");
  CUS(cudaMemcpyAsync(&bar, w.bar, sizeof(GridBar), cudaMemcpyDeviceToHost, st), "decode_static: barrier D2H");
  CUS(cudaStreamSynchronize(st), "decode_static");
  if (bar.error & 1u)
    return api_fail(WFST_ERR_TIMEOUT, "decode_static: a device-side grid barrier wait timed out; the call was abandoned");
  if (bar.error & 2u) return api_fail(WFST_ERR_CUDA, "decode_static: epsilon closure did not converge");
  if (bar.error & 4u)
    return api_fail(WFST_ERR_TIMEOUT, "decode_static: a recombination CAS loop gave up after its retry bound");
  // words of every lane; a copy error is reported only after the stream has
  // drained, so no copy is left running when the call returns
  cudaError_t copy_err = cudaSuccess;
  int32_t short_lane = -1;
  for (int32_t b = 0; b < B; b++) {
    const Result& r = res[b];
    const int32_t nw = r.ok ? r.n_words : 0;
    if (words && words_cap > 0 && nw > 0) {
      const int32_t k = std::min(nw, words_cap);
      const cudaError_t e = cudaMemcpyAsync(words + (size_t)b * words_cap, w.words + (size_t)b * wc,
                                            sizeof(int32_t) * k, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess && copy_err == cudaSuccess) copy_err = e;
    }
    if (word_lens) word_lens[b] = nw;
    if (scores) scores[b] = r.ok ? (double)r.score : -INFINITY;
    if (meta) {
      meta[3 * b + 0] = r.ok;
      meta[3 * b + 1] = r.reached_final;
      meta[3 * b + 2] = lanes[b].overflow;
    }
    if (lanes[b].overflow && short_lane < 0) short_lane = b;
  }
  const cudaError_t sync_err = cudaStreamSynchronize(st);
  drain.armed = false;
  if (copy_err != cudaSuccess) return api_cuda_fail(copy_err, "decode_static: words D2H");
  if (sync_err != cudaSuccess) return api_cuda_fail(sync_err, "decode_static");
  if (short_lane >= 0) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "decode_static: lane %d ran out of the region's winners log (%lld entries per lane; overflow bits %d); "
             "wfst_decode grows it",
             (int)short_lane, (long long)log_cap, (int)lanes[short_lane].overflow);
    return api_fail(WFST_ERR_CAPACITY, msg);
  }
  return WFST_OK;
}
