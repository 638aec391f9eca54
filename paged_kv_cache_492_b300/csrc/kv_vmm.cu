// Elastic page pool (Elastic KV Cache for LLM Serving, paperlayer.ai --
// section 3: one contiguous virtual range per pool whose physical backing is
// mapped and unmapped at the top of the range, so the attention kernels and
// every page id keep working while the pool grows or shrinks).
//
// A pool is one reserved virtual address range of max_bytes.  Growing maps
// one more physical allocation (cuMemCreate) directly above the mapped part;
// shrinking unmaps and releases whole allocations from the top.  Page p of a
// K or V pool lives at base + p * page_bytes for as long as it is mapped, so
// pages below the mapped size never move.  The driver's virtual memory calls
// are looked up at run time through the runtime (no link-time dependency on
// libcuda).
#include <cuda.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "kv_internal.h"

namespace kvb {
namespace {

struct DriverVmm {
  CUresult (*reserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
  CUresult (*addr_free)(CUdeviceptr, size_t) = nullptr;
  CUresult (*create)(CUmemGenericAllocationHandle*, size_t, const CUmemAllocationProp*,
                     unsigned long long) = nullptr;
  CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
  CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle,
                  unsigned long long) = nullptr;
  CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
  CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t) = nullptr;
  CUresult (*granularity)(size_t*, const CUmemAllocationProp*,
                          CUmemAllocationGranularity_flags) = nullptr;
  bool ok = false;
};

int load_vmm(DriverVmm* out) {
  static std::mutex mu;
  static DriverVmm d;
  static bool tried = false;
  std::lock_guard<std::mutex> lk(mu);
  if (!tried) {
    tried = true;
    auto get = [](const char* name, void** fn) {
      cudaDriverEntryPointQueryResult q;
      return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) ==
                 cudaSuccess &&
             q == cudaDriverEntryPointSuccess && *fn != nullptr;
    };
    d.ok = get("cuMemAddressReserve", reinterpret_cast<void**>(&d.reserve)) &&
           get("cuMemAddressFree", reinterpret_cast<void**>(&d.addr_free)) &&
           get("cuMemCreate", reinterpret_cast<void**>(&d.create)) &&
           get("cuMemRelease", reinterpret_cast<void**>(&d.release)) &&
           get("cuMemMap", reinterpret_cast<void**>(&d.map)) &&
           get("cuMemUnmap", reinterpret_cast<void**>(&d.unmap)) &&
           get("cuMemSetAccess", reinterpret_cast<void**>(&d.set_access)) &&
           get("cuMemGetAllocationGranularity", reinterpret_cast<void**>(&d.granularity));
  }
  if (!d.ok) return cuda_failed(cudaErrorNotSupported, "driver virtual memory entry points");
  *out = d;
  return KV_OK;
}

struct Chunk {
  CUmemGenericAllocationHandle handle;
  size_t offset, bytes;
};

struct VmmPool {
  DriverVmm drv;
  int device = 0;
  CUdeviceptr base = 0;
  size_t reserved = 0, granularity = 0, mapped = 0;
  std::vector<Chunk> chunks;  // bottom to top
  std::mutex mu;
};

CUmemAllocationProp device_prop(int device) {
  CUmemAllocationProp prop;
  memset(&prop, 0, sizeof prop);
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = device;
  return prop;
}

int driver_failed(CUresult r, const char* what) {
  char msg[96];
  snprintf(msg, sizeof msg, "%s returned CUresult %d", what, (int)r);
  return cuda_failed(cudaErrorUnknown, msg);
}

}  // namespace
}  // namespace kvb

using namespace kvb;

extern "C" {

int kv_vmm_pool_create(int device, size_t max_bytes, void** pool, void** base,
                       size_t* granularity) {
  if (!pool || !base || max_bytes == 0) return KV_EINVAL;
  *pool = nullptr;
  *base = nullptr;
  DriverVmm drv;
  int rc = load_vmm(&drv);
  if (rc) return rc;
  const CUmemAllocationProp prop = device_prop(device);
  size_t gran = 0;
  CUresult r = drv.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED);
  if (r != CUDA_SUCCESS || gran == 0) return driver_failed(r, "cuMemGetAllocationGranularity");
  const size_t reserved = align_up(max_bytes, gran);
  CUdeviceptr ptr = 0;
  r = drv.reserve(&ptr, reserved, gran, 0, 0);
  if (r != CUDA_SUCCESS) return driver_failed(r, "cuMemAddressReserve");
  VmmPool* p = new (std::nothrow) VmmPool();
  if (!p) {
    drv.addr_free(ptr, reserved);
    return KV_EINVAL;
  }
  p->drv = drv;
  p->device = device;
  p->base = ptr;
  p->reserved = reserved;
  p->granularity = gran;
  *pool = p;
  *base = reinterpret_cast<void*>(ptr);
  if (granularity) *granularity = gran;
  return KV_OK;
}

size_t kv_vmm_pool_mapped(void* pool) {
  if (!pool) return 0;
  VmmPool* p = static_cast<VmmPool*>(pool);
  std::lock_guard<std::mutex> lk(p->mu);
  return p->mapped;
}

int kv_vmm_pool_resize(void* pool, size_t bytes, size_t* mapped) {
  if (!pool) return KV_EINVAL;
  VmmPool* p = static_cast<VmmPool*>(pool);
  std::lock_guard<std::mutex> lk(p->mu);
  const DriverVmm& d = p->drv;
  const size_t target = align_up(bytes, p->granularity);
  if (target > p->reserved) return KV_EINVAL;
  if (target > p->mapped) {
    // grow: one physical allocation for the whole new slice, mapped on top
    const size_t add = target - p->mapped;
    const CUmemAllocationProp prop = device_prop(p->device);
    CUmemGenericAllocationHandle h;
    CUresult r = d.create(&h, add, &prop, 0);
    if (r != CUDA_SUCCESS) return driver_failed(r, "cuMemCreate");
    r = d.map(p->base + p->mapped, add, 0, h, 0);
    if (r != CUDA_SUCCESS) {
      d.release(h);
      return driver_failed(r, "cuMemMap");
    }
    CUmemAccessDesc acc;
    memset(&acc, 0, sizeof acc);
    acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc.location.id = p->device;
    acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    r = d.set_access(p->base + p->mapped, add, &acc, 1);
    if (r != CUDA_SUCCESS) {
      d.unmap(p->base + p->mapped, add);
      d.release(h);
      return driver_failed(r, "cuMemSetAccess");
    }
    p->chunks.push_back(Chunk{h, p->mapped, add});
    p->mapped = target;
  } else {
    // shrink: release whole slices from the top while they lie above target
    while (!p->chunks.empty() && p->chunks.back().offset >= target) {
      const Chunk c = p->chunks.back();
      CUresult r = d.unmap(p->base + c.offset, c.bytes);
      if (r != CUDA_SUCCESS) return driver_failed(r, "cuMemUnmap");
      r = d.release(c.handle);
      if (r != CUDA_SUCCESS) return driver_failed(r, "cuMemRelease");
      p->chunks.pop_back();
      p->mapped = c.offset;
    }
  }
  if (mapped) *mapped = p->mapped;
  return KV_OK;
}

int kv_vmm_pool_destroy(void* pool) {
  if (!pool) return KV_EINVAL;
  VmmPool* p = static_cast<VmmPool*>(pool);
  int rc = KV_OK;
  {
    std::lock_guard<std::mutex> lk(p->mu);
    const DriverVmm& d = p->drv;
    while (!p->chunks.empty()) {
      const Chunk c = p->chunks.back();
      if (d.unmap(p->base + c.offset, c.bytes) != CUDA_SUCCESS ||
          d.release(c.handle) != CUDA_SUCCESS)
        rc = driver_failed(CUDA_ERROR_UNKNOWN, "cuMemUnmap/cuMemRelease");
      p->chunks.pop_back();
    }
    if (d.addr_free(p->base, p->reserved) != CUDA_SUCCESS)
      rc = driver_failed(CUDA_ERROR_UNKNOWN, "cuMemAddressFree");
  }
  delete p;
  return rc;
}

}  // extern "C"
