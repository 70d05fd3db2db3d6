// wfst_vmm.cu — LazyRegions: per-lane device regions committed on demand
// through the CUDA driver's virtual memory management calls, reached with
// cudaGetDriverEntryPointByVersion (no link-time dependence on libcuda).
#include "wfst_vmm.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

namespace wfst {

namespace {

typedef CUresult (*FnReserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long);
typedef CUresult (*FnFree)(CUdeviceptr, size_t);
typedef CUresult (*FnCreate)(CUmemGenericAllocationHandle*, size_t, const CUmemAllocationProp*,
                             unsigned long long);
typedef CUresult (*FnRelease)(CUmemGenericAllocationHandle);
typedef CUresult (*FnMap)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long);
typedef CUresult (*FnUnmap)(CUdeviceptr, size_t);
typedef CUresult (*FnAccess)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t);
typedef CUresult (*FnGran)(size_t*, const CUmemAllocationProp*, CUmemAllocationGranularity_flags);

struct Driver {
  FnReserve reserve = nullptr;
  FnFree free = nullptr;
  FnCreate create = nullptr;
  FnRelease release = nullptr;
  FnMap map = nullptr;
  FnUnmap unmap = nullptr;
  FnAccess access = nullptr;
  FnGran gran = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F* fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p) {
    cudaGetLastError();
    return false;
  }
  *fn = reinterpret_cast<F>(p);
  return true;
}

const Driver& drv() {
  static Driver d;
  static std::once_flag once;
  std::call_once(once, [] {
    d.ok = entry("cuMemAddressReserve", &d.reserve) && entry("cuMemAddressFree", &d.free) &&
           entry("cuMemCreate", &d.create) && entry("cuMemRelease", &d.release) && entry("cuMemMap", &d.map) &&
           entry("cuMemUnmap", &d.unmap) && entry("cuMemSetAccess", &d.access) &&
           entry("cuMemGetAllocationGranularity", &d.gran);
  });
  return d;
}

CUmemAllocationProp prop_of(int device) {
  CUmemAllocationProp p = {};
  p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  p.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  p.location.id = device;
  return p;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t gcd(size_t a, size_t b) { return b ? gcd(b, a % b) : a; }

int fail(std::string* msg, const char* what, CUresult r) {
  if (msg) *msg = std::string(what) + " failed (CUDA driver error " + std::to_string((int)r) + ")";
  return (int)r;
}

}  // namespace

size_t LazyRegions::granularity(int device) {
  const Driver& d = drv();
  if (!d.ok) return 0;
  const CUmemAllocationProp p = prop_of(device);
  size_t g = 0;
  if (d.gran(&g, &p, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS) return 0;
  return g;
}

void LazyRegions::init(int device, int regions, size_t elem, int64_t stride_align) {
  release();
  device_ = device;
  regions_ = regions;
  elem_ = elem;
  gran_ = granularity(device);
  const size_t a = elem * (size_t)(stride_align > 0 ? stride_align : 1);
  align_bytes_ = gran_ ? gran_ / gcd(gran_, a) * a : a;  // lcm
}

int LazyRegions::map_all(CUdeviceptr base, size_t stride, std::string* msg) {
  const Driver& d = drv();
  CUmemAccessDesc acc = {};
  acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  acc.location.id = device_;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  for (size_t c = 0; c < chunks_.size(); c++) {
    const Chunk& k = chunks_[c];
    for (int r = 0; r < regions_; r++) {
      const CUdeviceptr at = base + (CUdeviceptr)((size_t)r * stride + k.offset);
      CUresult e = d.map(at, k.size, 0, k.h[(size_t)r], 0);
      if (e == CUDA_SUCCESS) e = d.access(at, k.size, &acc, 1);
      if (e != CUDA_SUCCESS) {
        // undo this call's mappings (chunks before c in full, chunk c up to r)
        for (size_t c2 = 0; c2 <= c; c2++)
          for (int r2 = 0; r2 < (c2 < c ? regions_ : r + 1); r2++)
            d.unmap(base + (CUdeviceptr)((size_t)r2 * stride + chunks_[c2].offset), chunks_[c2].size);
        return fail(msg, "cuMemMap", e);
      }
    }
  }
  return 0;
}

void LazyRegions::unmap_all(CUdeviceptr base, size_t stride) {
  const Driver& d = drv();
  for (const Chunk& k : chunks_)
    for (int r = 0; r < regions_; r++) d.unmap(base + (CUdeviceptr)((size_t)r * stride + k.offset), k.size);
}

int LazyRegions::reserve(int64_t stride_entries, std::string* msg) {
  const Driver& d = drv();
  if (!d.ok || !gran_) {
    if (msg) *msg = "CUDA virtual memory management is not available";
    return (int)CUDA_ERROR_NOT_SUPPORTED;
  }
  const size_t want = round_up((size_t)stride_entries * elem_, align_bytes_);
  if (want <= stride_) return 0;
  CUdeviceptr nb = 0;
  CUresult e = d.reserve(&nb, want * (size_t)regions_, gran_, 0, 0);
  if (e != CUDA_SUCCESS) return fail(msg, "cuMemAddressReserve", e);
  if (int rc = map_all(nb, want, msg)) {
    d.free(nb, want * (size_t)regions_);
    return rc;
  }
  if (base_) {
    unmap_all(base_, stride_);
    d.free(base_, stride_ * (size_t)regions_);
  }
  base_ = nb;
  stride_ = want;
  return 0;
}

int LazyRegions::commit(int64_t entries, std::string* msg) {
  const Driver& d = drv();
  const size_t need = round_up((size_t)entries * elem_, gran_ ? gran_ : 1);
  if (need <= committed_) return 0;
  if (need > stride_) {
    if (int rc = reserve((int64_t)(std::max(need, 2 * stride_) / elem_), msg)) return rc;
  }
  const size_t delta = need - committed_;
  const CUmemAllocationProp p = prop_of(device_);
  CUmemAccessDesc acc = {};
  acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  acc.location.id = device_;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  Chunk k{std::vector<CUmemGenericAllocationHandle>((size_t)regions_), committed_, delta};
  for (int r = 0; r < regions_; r++) {
    const CUdeviceptr at = base_ + (CUdeviceptr)((size_t)r * stride_ + committed_);
    CUresult e = d.create(&k.h[(size_t)r], delta, &p, 0);
    const bool made = e == CUDA_SUCCESS;
    if (made) e = d.map(at, delta, 0, k.h[(size_t)r], 0);
    if (e == CUDA_SUCCESS) e = d.access(at, delta, &acc, 1);
    if (e != CUDA_SUCCESS) {
      // undo this commit: regions before r in full, region r as far as it got
      for (int r2 = 0; r2 <= r; r2++) {
        if (r2 < r || made) d.unmap(base_ + (CUdeviceptr)((size_t)r2 * stride_ + committed_), delta);
        if (r2 < r || made) d.release(k.h[(size_t)r2]);
      }
      return fail(msg, made ? "cuMemMap" : "cuMemCreate", e);
    }
  }
  chunks_.push_back(std::move(k));
  committed_ = need;
  return 0;
}

void LazyRegions::release() {
  if (!regions_) return;
  const Driver& d = drv();
  if (base_) {
    unmap_all(base_, stride_);
    d.free(base_, stride_ * (size_t)regions_);
  }
  for (const Chunk& k : chunks_)
    for (CUmemGenericAllocationHandle h : k.h) d.release(h);
  chunks_.clear();
  base_ = 0;
  stride_ = 0;
  committed_ = 0;
  regions_ = 0;
}

}  // namespace wfst
