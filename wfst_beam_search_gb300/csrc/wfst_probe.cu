// wfst_probe.cu — wfst_probe_random_gather: a measurement kernel, not part
// of the decoder.  It reads random segments of a large caller-owned device
// table as fast as the memory system allows, so that a benchmark can state
// the device's ceiling for random accesses next to its copy bandwidth.  The
// decoder's traffic is random lines (recombination entries, arc rows), and
// such accesses are limited by how many the DRAM can serve per second, not
// by the bytes each one moves.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/wfst_gb300.h"

namespace wfst {
int api_fail(int code, const char* msg);
int api_cuda_fail(cudaError_t e, const char* what);
}  // namespace wfst

namespace {

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Group g of W consecutive threads reads one segment of W 16-byte words at
// a random segment-aligned index in [0, n16); every thread issues `loads`
// reads, four independent ones at a time.
template <int W>
__global__ void gather_kernel(const int4* __restrict__ buf, uint32_t nseg, int loads, uint32_t seed, int* sink) {
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t grp = tid / W, sub = tid % W;
  int acc = 0;
  for (int i = 0; i < loads; i += 4) {
    int4 v[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const uint32_t seg = mix32(grp * 2654435761u + (uint32_t)(i + k) * 40503u + seed) % nseg;
      v[k] = __ldcg(buf + (size_t)seg * W + sub);
    }
#pragma unroll
    for (int k = 0; k < 4; k++) acc += v[k].x ^ v[k].w;
  }
  if (acc == 0x7fffffff) *sink = acc;  // keeps the loads; practically never taken
}

}  // namespace

extern "C" int wfst_probe_random_gather(const void* table, int64_t table_bytes, int32_t seg_bytes, int32_t grid,
                                        int32_t loads_per_thread, int32_t seed, int32_t* sink, void* stream) {
  using namespace wfst;
  if (!table || !sink || grid < 1 || loads_per_thread < 4 || loads_per_thread % 4 != 0)
    return api_fail(WFST_ERR_INVALID_ARG, "probe_random_gather: bad argument");
  if (seg_bytes != 16 && seg_bytes != 64 && seg_bytes != 128)
    return api_fail(WFST_ERR_INVALID_ARG, "probe_random_gather: seg_bytes must be 16, 64 or 128");
  const int64_t nseg = table_bytes / seg_bytes;
  if (nseg < 1 || nseg > (int64_t)UINT32_MAX)
    return api_fail(WFST_ERR_INVALID_ARG, "probe_random_gather: the table must hold 1 .. 2^32-1 segments");
  if ((uintptr_t)table % 16 != 0) return api_fail(WFST_ERR_INVALID_ARG, "probe_random_gather: table not 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const int threads = 512;
  const auto* buf = static_cast<const int4*>(table);
  if (seg_bytes == 16) gather_kernel<1><<<grid, threads, 0, st>>>(buf, (uint32_t)nseg, loads_per_thread, (uint32_t)seed, sink);
  if (seg_bytes == 64) gather_kernel<4><<<grid, threads, 0, st>>>(buf, (uint32_t)nseg, loads_per_thread, (uint32_t)seed, sink);
  if (seg_bytes == 128) gather_kernel<8><<<grid, threads, 0, st>>>(buf, (uint32_t)nseg, loads_per_thread, (uint32_t)seed, sink);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? WFST_OK : api_cuda_fail(e, "probe_random_gather launch");
}
