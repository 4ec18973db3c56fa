// VMM-backed output workspace for lazy chunking.
//
// "Mosaic: Unlocking Long-Context Inference for Diffusion LLMs via Global Memory" (paper review,
// section 3, core component 4 "Global Memory Manager") and "扩散大语言模型内存优化：Mosaic系统
// 突破与实践" (section 3.1): reserve a contiguous virtual address range up front without physical
// memory, then bind physical pages to it as the actual demand grows, so buffers keep one address
// and fragmentation cannot occur. At the scale of this single operator that is the chunk output
// buffer: its virtual range is reserved for the largest output the caller may ever need and
// physical pages are bound only as far as the chunk sizes actually used, and can be released
// again when the demand falls.
//
// Built on the CUDA driver's virtual memory management (cuMemAddressReserve, cuMemCreate,
// cuMemMap, cuMemSetAccess, cuMemUnmap, cuMemRelease), reached through the runtime's
// driver-entry-point lookup so the library does not link the driver library directly.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/mosaic.h"
#include "status.h"

namespace {

struct VmmApi {
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

const VmmApi& vmm() {
  static VmmApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    auto get = [](const char* name, void** fn) {
      cudaDriverEntryPointQueryResult q;
      return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) ==
                 cudaSuccess &&
             q == cudaDriverEntryPointSuccess;
    };
    api.ok = get("cuMemAddressReserve", reinterpret_cast<void**>(&api.reserve)) &&
             get("cuMemAddressFree", reinterpret_cast<void**>(&api.free_va)) &&
             get("cuMemCreate", reinterpret_cast<void**>(&api.create)) &&
             get("cuMemRelease", reinterpret_cast<void**>(&api.release)) &&
             get("cuMemMap", reinterpret_cast<void**>(&api.map)) &&
             get("cuMemUnmap", reinterpret_cast<void**>(&api.unmap)) &&
             get("cuMemSetAccess", reinterpret_cast<void**>(&api.set_access)) &&
             get("cuMemGetAllocationGranularity", reinterpret_cast<void**>(&api.granularity));
  });
  return api;
}

mosaic_status ws_fail(mosaic_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  mosaic::set_last_error(buf);
  return s;
}

}  // namespace

struct mosaic_workspace {
  int device = 0;
  CUdeviceptr base = 0;
  size_t reserved = 0;
  size_t granule = 0;
  size_t bound = 0;
  CUmemAllocationProp prop = {};
  std::vector<std::pair<CUmemGenericAllocationHandle, size_t>> pieces;  // in address order
};

extern "C" {

mosaic_status mosaic_workspace_create(mosaic_workspace** out, int device, int64_t reserve_bytes) {
  if (!out) return ws_fail(MOSAIC_ERR_INVALID_ARG, "NULL out-pointer");
  *out = nullptr;
  if (reserve_bytes < 1) return ws_fail(MOSAIC_ERR_INVALID_ARG, "reserve_bytes must be >= 1");
  cudaError_t e = cudaSetDevice(device);
  if (e == cudaSuccess) e = cudaFree(nullptr);  // make the device's primary context current
  if (e != cudaSuccess) return ws_fail(MOSAIC_ERR_CUDA, "device %d: %s", device, cudaGetErrorString(e));
  const VmmApi& api = vmm();
  if (!api.ok) return ws_fail(MOSAIC_ERR_CUDA, "CUDA virtual memory management entry points not found");
  auto* ws = new mosaic_workspace();
  ws->device = device;
  ws->prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  ws->prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  ws->prop.location.id = device;
  CUresult r = api.granularity(&ws->granule, &ws->prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED);
  if (r != CUDA_SUCCESS || ws->granule == 0) {
    delete ws;
    return ws_fail(MOSAIC_ERR_CUDA, "cuMemGetAllocationGranularity failed (%d)", static_cast<int>(r));
  }
  ws->reserved = (static_cast<size_t>(reserve_bytes) + ws->granule - 1) / ws->granule * ws->granule;
  r = api.reserve(&ws->base, ws->reserved, ws->granule, 0, 0);
  if (r != CUDA_SUCCESS) {
    delete ws;
    return ws_fail(MOSAIC_ERR_CUDA, "cuMemAddressReserve of %zu bytes failed (%d)", ws->reserved,
                   static_cast<int>(r));
  }
  *out = ws;
  return MOSAIC_OK;
}

mosaic_status mosaic_workspace_bind(mosaic_workspace* ws, int64_t bytes, void** ptr) {
  if (!ws || !ptr) return ws_fail(MOSAIC_ERR_INVALID_ARG, "NULL workspace or out-pointer");
  if (bytes < 0) return ws_fail(MOSAIC_ERR_INVALID_ARG, "bytes < 0");
  const size_t need = (static_cast<size_t>(bytes) + ws->granule - 1) / ws->granule * ws->granule;
  if (need > ws->reserved)
    return ws_fail(MOSAIC_ERR_UNSUPPORTED, "%lld bytes exceed the %zu reserved",
                   static_cast<long long>(bytes), ws->reserved);
  if (need > ws->bound) {
    const VmmApi& api = vmm();
    const size_t size = need - ws->bound;
    CUmemGenericAllocationHandle h;
    CUresult r = api.create(&h, size, &ws->prop, 0);
    if (r != CUDA_SUCCESS)
      return ws_fail(MOSAIC_ERR_CUDA, "cuMemCreate of %zu bytes failed (%d)", size, static_cast<int>(r));
    r = api.map(ws->base + ws->bound, size, 0, h, 0);
    if (r != CUDA_SUCCESS) {
      api.release(h);
      return ws_fail(MOSAIC_ERR_CUDA, "cuMemMap failed (%d)", static_cast<int>(r));
    }
    CUmemAccessDesc access = {};
    access.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    access.location.id = ws->device;
    access.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    r = api.set_access(ws->base + ws->bound, size, &access, 1);
    if (r != CUDA_SUCCESS) {
      api.unmap(ws->base + ws->bound, size);
      api.release(h);
      return ws_fail(MOSAIC_ERR_CUDA, "cuMemSetAccess failed (%d)", static_cast<int>(r));
    }
    ws->pieces.emplace_back(h, size);
    ws->bound = need;
  }
  *ptr = reinterpret_cast<void*>(ws->base);
  return MOSAIC_OK;
}

mosaic_status mosaic_workspace_trim(mosaic_workspace* ws, int64_t keep_bytes) {
  if (!ws) return ws_fail(MOSAIC_ERR_INVALID_ARG, "NULL workspace");
  if (keep_bytes < 0) return ws_fail(MOSAIC_ERR_INVALID_ARG, "keep_bytes < 0");
  cudaSetDevice(ws->device);
  cudaError_t e = cudaDeviceSynchronize();  // nothing may still use the pages being unbound
  if (e != cudaSuccess) return ws_fail(MOSAIC_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
  const VmmApi& api = vmm();
  while (!ws->pieces.empty() && ws->bound - ws->pieces.back().second >= static_cast<size_t>(keep_bytes)) {
    const auto piece = ws->pieces.back();
    const CUdeviceptr at = ws->base + ws->bound - piece.second;
    if (api.unmap(at, piece.second) != CUDA_SUCCESS || api.release(piece.first) != CUDA_SUCCESS)
      return ws_fail(MOSAIC_ERR_CUDA, "unbinding %zu bytes failed", piece.second);
    ws->pieces.pop_back();
    ws->bound -= piece.second;
  }
  return MOSAIC_OK;
}

int64_t mosaic_workspace_bound_bytes(const mosaic_workspace* ws) {
  return ws ? static_cast<int64_t>(ws->bound) : -1;
}

int64_t mosaic_workspace_reserved_bytes(const mosaic_workspace* ws) {
  return ws ? static_cast<int64_t>(ws->reserved) : -1;
}

mosaic_status mosaic_workspace_destroy(mosaic_workspace* ws) {
  if (!ws) return MOSAIC_OK;
  mosaic_status st = mosaic_workspace_trim(ws, 0);
  if (st != MOSAIC_OK) return st;
  if (vmm().free_va(ws->base, ws->reserved) != CUDA_SUCCESS)
    return ws_fail(MOSAIC_ERR_CUDA, "cuMemAddressFree failed");
  delete ws;
  return MOSAIC_OK;
}

}  // extern "C"
