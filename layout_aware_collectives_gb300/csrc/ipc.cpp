// Peer memory of rank processes: export a buffer's allocation as a CUDA IPC
// handle, map a peer's allocation into this process, unmap it.
//
// With one process per rank, TIDE-RS reads every rank's per-parameter bf16
// gradients directly ("FSDP通信终局：TIDE零拷贝集合通信优化" §TIDE的设计思路): rank
// r's reduce-scatter kernel gets a pointer table whose entries for the other
// ranks are their gradient addresses mapped into r's address space.  These
// calls produce those addresses; the kernels are the library's single-rank
// reduce-scatter and placement, unchanged.
#include <cuda.h>  // driver-API types only; the entry point is fetched through the runtime
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "tide_internal.h"

namespace tide {
namespace {

static_assert(sizeof(cudaIpcMemHandle_t) == TIDE_IPC_HANDLE_BYTES, "IPC handle size");

using MemGetAddressRange = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
std::once_flag g_once;
MemGetAddressRange g_range = nullptr;

MemGetAddressRange address_range_fn() {
  std::call_once(g_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_range = (MemGetAddressRange)f;
    cudaGetLastError();
  });
  return g_range;
}

}  // namespace
}  // namespace tide

using namespace tide;

extern "C" {

tide_status_t tide_ipc_export(const void* ptr, uint8_t* handle, uint64_t* offset) {
  if (!ptr || !handle || !offset) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  MemGetAddressRange range = address_range_fn();
  if (!range) return set_error(TIDE_ERR_UNSUPPORTED, "the driver does not provide cuMemGetAddressRange");
  CUdeviceptr base = 0;
  size_t size = 0;
  const CUresult r = range(&base, &size, (CUdeviceptr)(uintptr_t)ptr);
  if (r != CUDA_SUCCESS || base == 0)
    return set_error(TIDE_ERR_INVALID_ARG, "pointer is not inside a device allocation (driver error " +
                                               std::to_string((int)r) + ")");
  cudaIpcMemHandle_t h;
  const cudaError_t e = cudaIpcGetMemHandle(&h, (void*)(uintptr_t)base);
  if (e != cudaSuccess) return cuda_fail(e, "cudaIpcGetMemHandle");
  std::memcpy(handle, &h, sizeof h);
  *offset = (uint64_t)((uintptr_t)ptr - (uintptr_t)base);
  return TIDE_OK;
}

tide_status_t tide_ipc_open(const uint8_t* handle, void** base) {
  if (!handle || !base) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  cudaIpcMemHandle_t h;
  std::memcpy(&h, handle, sizeof h);
  *base = nullptr;
  const cudaError_t e = cudaIpcOpenMemHandle(base, h, cudaIpcMemLazyEnablePeerAccess);
  if (e != cudaSuccess) return cuda_fail(e, "cudaIpcOpenMemHandle");
  return TIDE_OK;
}

tide_status_t tide_ipc_close(void* base) {
  if (!base) return set_error(TIDE_ERR_INVALID_ARG, "NULL argument");
  const cudaError_t e = cudaIpcCloseMemHandle(base);
  if (e != cudaSuccess) return cuda_fail(e, "cudaIpcCloseMemHandle");
  return TIDE_OK;
}

}  // extern "C"
