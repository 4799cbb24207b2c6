// Host memory for the cold KV history, mapped into the GPU's own page tables.
//
// The full history of an offloaded request stays in host memory and the
// attention reads its selected rows over the host link ("双卡RTX4090跑通
// Qwen3-Next：8并发满血长上下文实测", section "显存账本：热缓存卸载省下约84%":
// full history in pinned host memory, missing blocks brought back on demand).
// Pinned memory made by registering ordinary pages is reached, on an
// NVLink-C2C (Grace) system, through address translation services: every
// 64 KiB host page the GPU touches is translated through the CPU's page
// tables.  This allocator instead creates the physical pages on a host NUMA
// node with the driver's virtual-memory API and maps them, in 2 MiB pieces,
// into one virtual range that is entered in the GPU's own page tables (and
// in the CPU's, so the host reads and writes it at the same address).  The
// GPU then translates a whole 2 MiB piece with one entry.
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

struct VmmDriver {
  decltype(&cuMemGetAllocationGranularity) granularity = nullptr;
  decltype(&cuMemAddressReserve) reserve = nullptr;
  decltype(&cuMemAddressFree) address_free = nullptr;
  decltype(&cuMemCreate) create = nullptr;
  decltype(&cuMemRelease) release = nullptr;
  decltype(&cuMemMap) map = nullptr;
  decltype(&cuMemUnmap) unmap = nullptr;
  decltype(&cuMemSetAccess) set_access = nullptr;
  bool ok = false;
};

template <class F>
bool driver_entry(const char* name, F* out) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  *out = reinterpret_cast<F>(fn);
  return true;
}

const VmmDriver& vmm() {
  static const VmmDriver d = [] {
    VmmDriver v;
    v.ok = driver_entry("cuMemGetAllocationGranularity", &v.granularity) &&
           driver_entry("cuMemAddressReserve", &v.reserve) &&
           driver_entry("cuMemAddressFree", &v.address_free) &&
           driver_entry("cuMemCreate", &v.create) && driver_entry("cuMemRelease", &v.release) &&
           driver_entry("cuMemMap", &v.map) && driver_entry("cuMemUnmap", &v.unmap) &&
           driver_entry("cuMemSetAccess", &v.set_access);
    return v;
  }();
  return d;
}

struct Mapping {
  size_t bytes;    // mapped bytes (a multiple of the granularity)
  int device;      // device whose page tables hold the range
};

std::mutex g_mu;
std::map<uintptr_t, Mapping> g_maps;   // base address -> mapping

}  // namespace

bool host_alloc_covers(const void* p, int64_t bytes, int device) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_maps.upper_bound(a);
  if (it == g_maps.begin()) return false;
  --it;
  return it->second.device == device && bytes >= 0 &&
         a + (uint64_t)bytes <= it->first + it->second.bytes;
}

}  // namespace qsa

using namespace qsa;

extern "C" qsa_status_t qsa_host_alloc(int32_t device, int32_t numa_node, int64_t bytes, void** out) {
  if (!out) return set_last_error(QSA_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  if (bytes <= 0) return set_last_error(QSA_ERR_INVALID_ARG, "bytes must be positive");
  const VmmDriver& d = vmm();
  if (!d.ok) return set_last_error(QSA_ERR_CUDA, "the driver lacks the virtual-memory API");
  DeviceGuard guard(device);
  if (guard.status() != cudaSuccess) return set_last_error(QSA_ERR_INVALID_ARG, "bad device");
  cudaError_t e = cudaFree(nullptr);   // the device's context exists from here on
  if (e != cudaSuccess) return set_last_error(QSA_ERR_CUDA, cudaGetErrorString(e));
  if (numa_node < 0) {
    int node = -1;
    if (cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, device) != cudaSuccess) {
      cudaGetLastError();
      node = -1;
    }
    numa_node = node < 0 ? 0 : node;
  }
  CUmemAllocationProp prop{};
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
  prop.location.id = numa_node;
  size_t gran = 0;
  CUresult r = d.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED);
  if (r != CUDA_SUCCESS || gran == 0)
    return set_last_error(QSA_ERR_CUDA, "host NUMA memory is not available to this device");
  const size_t total = ((size_t)bytes + gran - 1) / gran * gran;
  const size_t chunk = ((size_t)1 << 30) / gran * gran > 0 ? ((size_t)1 << 30) / gran * gran : gran;
  CUdeviceptr va = 0;
  r = d.reserve(&va, total, gran, 0, 0);
  if (r != CUDA_SUCCESS) return set_last_error(QSA_ERR_CUDA, "reserving the virtual range");
  size_t mapped = 0;
  for (; mapped < total; mapped += chunk) {
    const size_t sz = total - mapped < chunk ? total - mapped : chunk;
    CUmemGenericAllocationHandle h;
    r = d.create(&h, sz, &prop, 0);
    if (r != CUDA_SUCCESS) break;
    r = d.map(va + mapped, sz, 0, h, 0);
    d.release(h);   // the mapping keeps the pages alive
    if (r != CUDA_SUCCESS) break;
  }
  if (r == CUDA_SUCCESS) {
    CUmemAccessDesc acc[2] = {};
    acc[0].location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc[0].location.id = device;
    acc[0].flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    acc[1].location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
    acc[1].location.id = numa_node;
    acc[1].flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    r = d.set_access(va, total, acc, 2);
  }
  if (r != CUDA_SUCCESS) {
    for (size_t off = 0; off < mapped && off < total; off += chunk)
      d.unmap(va + off, total - off < chunk ? total - off : chunk);
    d.address_free(va, total);
    return set_last_error(r == CUDA_ERROR_OUT_OF_MEMORY ? QSA_ERR_CAPACITY : QSA_ERR_CUDA,
                          "creating or mapping host NUMA memory");
  }
  {
    std::lock_guard<std::mutex> lock(g_mu);
    g_maps[(uintptr_t)va] = Mapping{total, device};
  }
  *out = reinterpret_cast<void*>(va);
  return set_last_error(QSA_OK, "");
}

extern "C" qsa_status_t qsa_host_free(void* ptr) {
  if (!ptr) return set_last_error(QSA_OK, "");
  Mapping m{};
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_maps.find(reinterpret_cast<uintptr_t>(ptr));
    if (it == g_maps.end())
      return set_last_error(QSA_ERR_INVALID_ARG, "pointer was not returned by qsa_host_alloc");
    m = it->second;
    g_maps.erase(it);
  }
  const VmmDriver& d = vmm();
  CUresult r = d.unmap(reinterpret_cast<CUdeviceptr>(ptr), m.bytes);
  CUresult r2 = d.address_free(reinterpret_cast<CUdeviceptr>(ptr), m.bytes);
  if (r != CUDA_SUCCESS || r2 != CUDA_SUCCESS)
    return set_last_error(QSA_ERR_CUDA, "unmapping host NUMA memory");
  return set_last_error(QSA_OK, "");
}
