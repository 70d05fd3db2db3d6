// wfst_preslice.cu — blank-skip frame pre-slicing, a pre-pass outside the
// decoder ("GPU WFST Beam-Search Decoder", §3 Decoding Semantics: frames
// whose blank posterior passes a threshold, 0.98 by default, are removed
// before the search, in the WeNet manner, not inside it; skipping inside the
// search would be wrong on graphs whose states do not all carry a blank
// self-loop).
//
// A frame t < lens[b] of lane b is dropped iff its blank log-posterior is
// above log(threshold): lp[b, t, blank] > lthr, where lthr is log(threshold)
// computed in double and rounded once to fp32, and lp is widened exactly to
// fp32.  The kept rows are packed, in order, into out[b, 0 .. out_lens[b]).
//
// Two kernels, both bound by HBM bandwidth:
//   keep_scan: one CTA per lane reads the blank column (one element per
//     frame), flags the kept frames and writes frame_map[b, i] = source frame
//     of kept row i (a CTA-wide scan over chunks of kThreads frames; -1 past
//     the kept count) and out_lens[b];
//   copy_rows: one warp per output row copies the kept row, 16 bytes per
//     lane when the source and destination rows are 16-byte aligned, else
//     element by element; rows past out_lens[b] are left untouched.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/wfst_gb300.h"

namespace wfst {
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
}  // namespace wfst

namespace {

constexpr int kScanThreads = 512;
constexpr int kCopyWarps = 8;

template <typename LP>
__device__ __forceinline__ float widen(LP v);
template <>
__device__ __forceinline__ float widen<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen<__half>(__half v) { return __half2float(v); }

template <typename LP>
__global__ void __launch_bounds__(kScanThreads) keep_scan(const LP* __restrict__ lp, int64_t stride_b,
                                                          int64_t stride_t, int32_t blank, float lthr,
                                                          const int32_t* __restrict__ lens, int32_t T,
                                                          int32_t* __restrict__ frame_map,
                                                          int32_t* __restrict__ out_lens) {
  __shared__ int32_t warp_tot[kScanThreads / 32];
  __shared__ int32_t base;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t len = min(max(lens[b], 0), T);
  const LP* row0 = lp + (int64_t)b * stride_b + blank;
  int32_t* map = frame_map + (int64_t)b * T;
  if (tid == 0) base = 0;
  __syncthreads();
  for (int32_t t0 = 0; t0 < T; t0 += kScanThreads) {
    const int32_t t = t0 + tid;
    bool keep = false;
    if (t < len) keep = !(widen<LP>(row0[(int64_t)t * stride_t]) > lthr);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    int32_t before = base;
    for (int k = 0; k < warp; k++) before += warp_tot[k];
    if (keep) map[before + __popc(m & ((1u << lane) - 1u))] = t;
    __syncthreads();
    if (tid == 0) {
      int32_t tot = 0;
      for (int k = 0; k < kScanThreads / 32; k++) tot += warp_tot[k];
      base += tot;
    }
    __syncthreads();
  }
  const int32_t kept = base;
  for (int32_t i = kept + tid; i < T; i += kScanThreads) map[i] = -1;
  if (tid == 0) out_lens[b] = kept;
}

__global__ void __launch_bounds__(kCopyWarps * 32) copy_rows(const unsigned char* __restrict__ lp, int64_t sb_bytes,
                                                             int64_t st_bytes, int64_t row_bytes, int32_t B,
                                                             int32_t T, const int32_t* __restrict__ frame_map,
                                                             const int32_t* __restrict__ out_lens,
                                                             unsigned char* __restrict__ out, int esz) {
  const int lane = threadIdx.x & 31;
  const int64_t nrows = (int64_t)B * T;
  const int64_t wstride = (int64_t)gridDim.x * kCopyWarps;
  for (int64_t r = (int64_t)blockIdx.x * kCopyWarps + (threadIdx.x >> 5); r < nrows; r += wstride) {
    const int32_t b = (int32_t)(r / T), i = (int32_t)(r % T);
    if (i >= out_lens[b]) continue;
    const int32_t t = frame_map[r];
    const unsigned char* src = lp + (int64_t)b * sb_bytes + (int64_t)t * st_bytes;
    unsigned char* dst = out + r * row_bytes;
    if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)row_bytes) & 15) == 0) {
      const int4* s4 = reinterpret_cast<const int4*>(src);
      int4* d4 = reinterpret_cast<int4*>(dst);
      for (int64_t k = lane; k < row_bytes / 16; k += 32) d4[k] = __ldg(s4 + k);
    } else if (esz == 4) {
      const float* s = reinterpret_cast<const float*>(src);
      float* d = reinterpret_cast<float*>(dst);
      for (int64_t k = lane; k < row_bytes / 4; k += 32) d[k] = __ldg(s + k);
    } else {
      const unsigned short* s = reinterpret_cast<const unsigned short*>(src);
      unsigned short* d = reinterpret_cast<unsigned short*>(dst);
      for (int64_t k = lane; k < row_bytes / 2; k += 32) d[k] = __ldg(s + k);
    }
  }
}

}  // namespace

extern "C" int wfst_blank_skip(const void* log_probs, int32_t dtype, int64_t stride_b, int64_t stride_t,
                               int32_t vocab_size, int32_t blank_id, float threshold, const int32_t* lens,
                               int32_t B, int32_t T, void* out, int32_t* out_lens, int32_t* frame_map,
                               void* stream) {
  using namespace wfst;
  if (B < 0 || T < 0) return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: B and T must be >= 0");
  if (B == 0 || T == 0) return WFST_OK;
  if (!log_probs || !lens || !out || !out_lens || !frame_map)
    return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: NULL argument");
  if (dtype != WFST_F32 && dtype != WFST_F16) return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: bad dtype");
  if (vocab_size < 1 || blank_id < 0 || blank_id >= vocab_size)
    return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: blank_id must lie in [0, vocab_size)");
  if (stride_t < vocab_size || stride_b < 0)
    return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: stride_t must be >= vocab_size and stride_b >= 0");
  if (!(threshold > 0.f)) return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: threshold must be > 0");
  for (const void* p : {log_probs, (const void*)lens, (const void*)out, (const void*)out_lens,
                        (const void*)frame_map}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: every array must be device memory");
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
      return api_fail(WFST_ERR_INVALID_ARG, "blank_skip: every array must be device memory");
  }
  cudaStream_t st = (cudaStream_t)stream;
  const float lthr = (float)std::log((double)threshold);
  const int esz = dtype == WFST_F16 ? 2 : 4;
  if (dtype == WFST_F16)
    keep_scan<__half><<<B, kScanThreads, 0, st>>>(reinterpret_cast<const __half*>(log_probs), stride_b,
                                                   stride_t, blank_id, lthr, lens, T, frame_map, out_lens);
  else
    keep_scan<float><<<B, kScanThreads, 0, st>>>(reinterpret_cast<const float*>(log_probs), stride_b, stride_t,
                                                 blank_id, lthr, lens, T, frame_map, out_lens);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return api_cuda_fail(e, "blank_skip: keep_scan launch");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = (int64_t)B * T;
  const int64_t want = (rows + kCopyWarps - 1) / kCopyWarps;
  const int grid = (int)std::min<int64_t>(want, (int64_t)std::max(sms, 1) * 8);
  copy_rows<<<grid, kCopyWarps * 32, 0, st>>>(reinterpret_cast<const unsigned char*>(log_probs),
                                               stride_b * esz, stride_t * esz, (int64_t)vocab_size * esz, B, T,
                                               frame_map, out_lens, reinterpret_cast<unsigned char*>(out), esz);
  e = cudaGetLastError();
  if (e != cudaSuccess) return api_cuda_fail(e, "blank_skip: copy_rows launch");
  return WFST_OK;
}
