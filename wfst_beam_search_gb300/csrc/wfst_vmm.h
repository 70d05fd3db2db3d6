// wfst_vmm.h — equal per-lane regions of device virtual address space whose
// physical memory is committed on demand (CUDA virtual memory management).
//
// "GPU WFST Beam-Search Decoder" §6.2 (lazily committed regions): the
// decoder reserves worst-case address ranges for its growing tables and
// backs only what the search reaches.  Here a table of R regions (lanes, or
// lane x frame parity) keeps one stride between regions and commits the
// same number of entries in each; committing more maps new physical memory
// after what each region already holds, so addresses and contents stay as
// they are.  Only when a commit passes the stride is a larger range
// reserved, and the physical memory already committed is mapped into it
// (no copy).
#pragma once
#include <cuda.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

namespace wfst {

class LazyRegions {
 public:
  LazyRegions() = default;
  LazyRegions(const LazyRegions&) = delete;
  LazyRegions& operator=(const LazyRegions&) = delete;
  ~LazyRegions() { release(); }

  // R regions of `elem`-byte entries on `device`; the stride between regions
  // is a multiple of `stride_align` entries (so that tables indexed alike
  // can share one stride).  Nothing is reserved yet.
  void init(int device, int regions, size_t elem, int64_t stride_align);
  // Reserve address space for `stride_entries` per region (rounded up); a
  // larger stride than the current one remaps the committed memory.
  // Returns 0, or a CUDA driver error with *msg set.
  int reserve(int64_t stride_entries, std::string* msg);
  // Commit at least `entries` per region (rounded up to the allocation
  // granularity), reserving a larger stride first when needed.
  int commit(int64_t entries, std::string* msg);
  void release();

  void* base() const { return reinterpret_cast<void*>(base_); }
  int64_t stride_entries() const { return elem_ ? (int64_t)(stride_ / elem_) : 0; }
  int64_t committed_entries() const { return elem_ ? (int64_t)(committed_ / elem_) : 0; }
  size_t reserved_bytes() const { return stride_ * (size_t)regions_; }
  size_t committed_bytes() const { return committed_ * (size_t)regions_; }
  bool active() const { return regions_ > 0; }

  // The allocation granularity of `device` (0 if VMM is unavailable).
  static size_t granularity(int device);

 private:
  struct Chunk {
    std::vector<CUmemGenericAllocationHandle> h;  // one physical allocation per region (a mapping
                                                  // always starts at offset 0 of its allocation)
    size_t offset;                                // offset inside each region
    size_t size;                                  // bytes per region
  };
  int map_all(CUdeviceptr base, size_t stride, std::string* msg);
  void unmap_all(CUdeviceptr base, size_t stride);

  int device_ = 0;
  int regions_ = 0;
  size_t elem_ = 0;
  size_t align_bytes_ = 0;  // stride alignment: lcm of the granularity and stride_align entries
  size_t gran_ = 0;
  CUdeviceptr base_ = 0;
  size_t stride_ = 0;       // bytes between regions (reserved per region)
  size_t committed_ = 0;    // bytes committed per region
  std::vector<Chunk> chunks_;
};

}  // namespace wfst
