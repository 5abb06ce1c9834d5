// Demand-mapped device arena for KV caches (hipfire, "QSA sparse attention
// and the VMM KV backend", section 04: reserve virtual address space for the
// longest context up front, back it with physical memory only as the cache
// grows, and keep one stable base pointer, so descriptors and captured work
// that hold addresses inside the arena stay valid while it grows).
//
// Host code only.  The driver's virtual-memory calls (reserve, create,
// map, set access) are reached through the runtime's driver entry-point
// query, so the library needs no link against the driver library.  Pages are
// mapped in whole allocation-granularity chunks and never unmapped while the
// arena lives; destroy() unmaps, releases and frees everything.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <new>
#include <vector>

#include "qsa_internal.cuh"

struct qsa_arena {
  int device = 0;
  CUdeviceptr base = 0;
  uint64_t reserved = 0;
  uint64_t mapped = 0;
  uint64_t granularity = 0;
  std::vector<CUmemGenericAllocationHandle> handles;
  std::vector<uint64_t> sizes;
  std::mutex lock;
};

namespace qsa {

namespace {

struct Vmm {
  PFN_cuMemAddressReserve_v10020 reserve = nullptr;
  PFN_cuMemAddressFree_v10020 free_va = nullptr;
  PFN_cuMemCreate_v10020 create = nullptr;
  PFN_cuMemRelease_v10020 release = nullptr;
  PFN_cuMemMap_v10020 map = nullptr;
  PFN_cuMemUnmap_v10020 unmap = nullptr;
  PFN_cuMemSetAccess_v10020 set_access = nullptr;
  PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F* out) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !f)
    return false;
  *out = reinterpret_cast<F>(f);
  return true;
}

const Vmm& vmm() {
  static Vmm v;
  static std::once_flag once;
  std::call_once(once, [] {
    v.ok = entry("cuMemAddressReserve", &v.reserve) && entry("cuMemAddressFree", &v.free_va) &&
           entry("cuMemCreate", &v.create) && entry("cuMemRelease", &v.release) && entry("cuMemMap", &v.map) &&
           entry("cuMemUnmap", &v.unmap) && entry("cuMemSetAccess", &v.set_access) &&
           entry("cuMemGetAllocationGranularity", &v.granularity);
  });
  return v;
}

CUmemAllocationProp device_prop(int device) {
  CUmemAllocationProp prop = {};
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = device;
  return prop;
}

}  // namespace

// Status-returning bodies of the C entry points (qsa_api.cu adds the error text).
qsa_status arena_create(int32_t device, uint64_t reserve_bytes, qsa_arena** out, const char** why) {
  *out = nullptr;
  const Vmm& v = vmm();
  if (!v.ok) {
    *why = "the driver's virtual-memory entry points are unavailable";
    return QSA_ERR_CUDA;
  }
  if (cudaSetDevice(device) != cudaSuccess || cudaFree(nullptr) != cudaSuccess) {
    *why = "no usable CUDA device";
    return QSA_ERR_CUDA;
  }
  const CUmemAllocationProp prop = device_prop(device);
  size_t gran = 0;
  if (v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED) != CUDA_SUCCESS || gran == 0) {
    *why = "cuMemGetAllocationGranularity failed";
    return QSA_ERR_CUDA;
  }
  qsa_arena* a = new (std::nothrow) qsa_arena();
  if (!a) {
    *why = "out of host memory";
    return QSA_ERR_CUDA;
  }
  a->device = device;
  a->granularity = gran;
  a->reserved = (reserve_bytes + gran - 1) / gran * gran;
  if (v.reserve(&a->base, a->reserved, gran, 0, 0) != CUDA_SUCCESS) {
    delete a;
    *why = "cuMemAddressReserve failed";
    return QSA_ERR_CUDA;
  }
  *out = a;
  return QSA_OK;
}

qsa_status arena_ensure(qsa_arena* a, uint64_t bytes, const char** why) {
  const Vmm& v = vmm();
  std::lock_guard<std::mutex> g(a->lock);
  if (bytes <= a->mapped) return QSA_OK;
  if (bytes > a->reserved) {
    *why = "more bytes than the arena reserved";
    return QSA_ERR_INVALID_ARG;
  }
  const uint64_t target = (bytes + a->granularity - 1) / a->granularity * a->granularity;
  const uint64_t size = target - a->mapped;
  const CUmemAllocationProp prop = device_prop(a->device);
  CUmemGenericAllocationHandle h = 0;
  if (v.create(&h, size, &prop, 0) != CUDA_SUCCESS) {
    *why = "cuMemCreate failed (out of device memory?)";
    return QSA_ERR_CUDA;
  }
  if (v.map(a->base + a->mapped, size, 0, h, 0) != CUDA_SUCCESS) {
    v.release(h);
    *why = "cuMemMap failed";
    return QSA_ERR_CUDA;
  }
  CUmemAccessDesc acc = {};
  acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  acc.location.id = a->device;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  if (v.set_access(a->base + a->mapped, size, &acc, 1) != CUDA_SUCCESS) {
    v.unmap(a->base + a->mapped, size);
    v.release(h);
    *why = "cuMemSetAccess failed";
    return QSA_ERR_CUDA;
  }
  a->handles.push_back(h);
  a->sizes.push_back(size);
  a->mapped = target;
  return QSA_OK;
}

qsa_status arena_destroy(qsa_arena* a, const char** why) {
  const Vmm& v = vmm();
  qsa_status s = QSA_OK;
  // Work still in flight may use the arena.
  if (cudaSetDevice(a->device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    *why = "device synchronize failed before unmapping";
    s = QSA_ERR_CUDA;
  }
  uint64_t off = 0;
  for (size_t i = 0; i < a->handles.size(); ++i) {
    if (v.unmap(a->base + off, a->sizes[i]) != CUDA_SUCCESS || v.release(a->handles[i]) != CUDA_SUCCESS) {
      *why = "cuMemUnmap / cuMemRelease failed";
      s = QSA_ERR_CUDA;
    }
    off += a->sizes[i];
  }
  if (a->base && v.free_va(a->base, a->reserved) != CUDA_SUCCESS) {
    *why = "cuMemAddressFree failed";
    s = QSA_ERR_CUDA;
  }
  delete a;
  return s;
}

void* arena_base(const qsa_arena* a) { return reinterpret_cast<void*>(a->base); }
uint64_t arena_mapped(const qsa_arena* a) { return a->mapped; }
uint64_t arena_reserved(const qsa_arena* a) { return a->reserved; }
uint64_t arena_granularity(const qsa_arena* a) { return a->granularity; }

}  // namespace qsa
