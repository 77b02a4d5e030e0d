// One virtual-address table per layer spanning device memory and host memory
// ("Running 125B MoE on Two 32 GB Cards", section 4.2 "One table that spans
// VRAM and host RAM": cuMemAddressReserve, cuMemCreate on the device and with
// CU_MEM_LOCATION_TYPE_HOST_NUMA on the host, cuMemMap of the two side by side).
//
// Layer l's table starts at va + l * (P + Hs): P bytes of device rows (the
// pool slots), then Hs bytes of host rows (the backing store), each part
// rounded up to the allocation granularity.  Each part is its own allocation
// (cuMemMap maps whole allocations).  The device gets read/write access to the
// whole range and the CPU to the host parts, so the host writes weights
// through the same addresses the kernels read.  The driver entry points come
// from the runtime, so the library does not link libcuda.

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "internal.cuh"

namespace moe {

namespace {

struct VmmApi {
  decltype(&cuMemAddressReserve) reserve = nullptr;
  decltype(&cuMemAddressFree) addr_free = nullptr;
  decltype(&cuMemCreate) create = nullptr;
  decltype(&cuMemRelease) release = nullptr;
  decltype(&cuMemMap) map = nullptr;
  decltype(&cuMemUnmap) unmap = nullptr;
  decltype(&cuMemSetAccess) set_access = nullptr;
  decltype(&cuMemGetAllocationGranularity) granularity = nullptr;
  decltype(&cuGetErrorString) err_str = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F* fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr) {
    cudaGetLastError();
    return false;
  }
  *fn = reinterpret_cast<F>(p);
  return true;
}

const VmmApi& api() {
  static VmmApi a;
  static bool tried = false;
  if (!tried) {
    tried = true;
    a.ok = entry("cuMemAddressReserve", &a.reserve) && entry("cuMemAddressFree", &a.addr_free) &&
           entry("cuMemCreate", &a.create) && entry("cuMemRelease", &a.release) && entry("cuMemMap", &a.map) &&
           entry("cuMemUnmap", &a.unmap) && entry("cuMemSetAccess", &a.set_access) &&
           entry("cuMemGetAllocationGranularity", &a.granularity) && entry("cuGetErrorString", &a.err_str);
  }
  return a;
}

std::string cu_msg(const VmmApi& a, const char* what, CUresult r) {
  const char* m = nullptr;
  if (a.err_str) a.err_str(r, &m);
  return std::string(what) + ": " + (m ? m : "CUDA driver error " + std::to_string((int)r));
}

size_t round_up(size_t v, size_t g) { return (v + g - 1) / g * g; }

}  // namespace

bool vmm_table_create(int device, int host_numa, int layers, size_t pool_bytes, size_t host_bytes, VmmTable* t,
                      std::string* err) {
  *t = VmmTable{};
  const VmmApi& a = api();
  if (!a.ok) {
    *err = "the CUDA driver does not provide the virtual memory management entry points";
    return false;
  }
  CUmemAllocationProp pd = {};
  pd.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  pd.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  pd.location.id = device;
  CUmemAllocationProp ph = {};
  ph.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  ph.location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
  ph.location.id = host_numa < 0 ? 0 : host_numa;
  size_t gd = 0, gh = 0;
  CUresult r = a.granularity(&gd, &pd, CU_MEM_ALLOC_GRANULARITY_MINIMUM);
  if (r == CUDA_SUCCESS) r = a.granularity(&gh, &ph, CU_MEM_ALLOC_GRANULARITY_MINIMUM);
  if (r != CUDA_SUCCESS) {
    *err = cu_msg(a, "cuMemGetAllocationGranularity", r);
    return false;
  }
  const size_t g = gd > gh ? gd : gh;
  t->pool_part = round_up(pool_bytes > 0 ? pool_bytes : 1, g);
  t->host_part = round_up(host_bytes > 0 ? host_bytes : 1, g);
  t->pitch = t->pool_part + t->host_part;
  t->bytes = t->pitch * (size_t)layers;
  auto undo = [&](const std::string& m) {
    *err = m;
    vmm_table_destroy(t);
    return false;
  };
  r = a.reserve(&t->va, t->bytes, g, 0, 0);
  if (r != CUDA_SUCCESS) {
    t->va = 0;
    return undo(cu_msg(a, "cuMemAddressReserve", r));
  }
  t->hdev.assign(layers, 0ull);
  t->hhost.assign(layers, 0ull);
  t->dev_mapped.assign(layers, 0);
  t->host_mapped.assign(layers, 0);
  for (int l = 0; l < layers; ++l) {
    const CUdeviceptr base = t->va + (CUdeviceptr)((size_t)l * t->pitch);
    CUmemGenericAllocationHandle h = 0;
    r = a.create(&h, t->pool_part, &pd, 0);
    if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemCreate (device rows)", r));
    t->hdev[l] = h;
    r = a.map(base, t->pool_part, 0, h, 0);
    if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemMap (device rows)", r));
    t->dev_mapped[l] = 1;
    r = a.create(&h, t->host_part, &ph, 0);
    if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemCreate (host rows, CU_MEM_LOCATION_TYPE_HOST_NUMA)", r));
    t->hhost[l] = h;
    r = a.map(base + t->pool_part, t->host_part, 0, h, 0);
    if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemMap (host rows)", r));
    t->host_mapped[l] = 1;
  }
  CUmemAccessDesc dacc = {};
  dacc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  dacc.location.id = device;
  dacc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  r = a.set_access(t->va, t->bytes, &dacc, 1);
  if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemSetAccess (device)", r));
  CUmemAccessDesc hacc = {};
  hacc.location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
  hacc.location.id = ph.location.id;
  hacc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  for (int l = 0; l < layers; ++l) {
    r = a.set_access(t->va + (CUdeviceptr)((size_t)l * t->pitch + t->pool_part), t->host_part, &hacc, 1);
    if (r != CUDA_SUCCESS) return undo(cu_msg(a, "cuMemSetAccess (host rows for the CPU)", r));
  }
  return true;
}

void vmm_table_destroy(VmmTable* t) {
  const VmmApi& a = api();
  if (!a.ok) return;
  for (size_t l = 0; l < t->hdev.size(); ++l) {
    const CUdeviceptr base = t->va + (CUdeviceptr)(l * t->pitch);
    if (t->dev_mapped[l]) a.unmap(base, t->pool_part);
    if (t->host_mapped[l]) a.unmap(base + t->pool_part, t->host_part);
    if (t->hdev[l]) a.release(t->hdev[l]);
    if (t->hhost[l]) a.release(t->hhost[l]);
  }
  if (t->va) a.addr_free(t->va, t->bytes);
  *t = VmmTable{};
}

}  // namespace moe
