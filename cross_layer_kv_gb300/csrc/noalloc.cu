// fkv_decode_attn_noalloc: decode attention for callers that cannot allocate
// device memory themselves.
//
// Some callers have no way to hand the library a workspace buffer: a host
// process whose device memory is entirely reserved by its own pool allocator,
// or a plugin interface that passes only the operands of one operation.
// cudaMalloc is not an option there either, since it synchronises the device
// and can fail once memory is exhausted.  This entry point therefore runs the
// same split + merge kernels as fkv_decode_attn with their partial results
// kept in a fixed-size array in the library's own device memory.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds kNoAllocScratchBytes of it until the process exits.  Host
// code must not hand its name to a kernel (on the host it is only a stand-in
// symbol); its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.  Make that first call before any stream capture.
//
// Every call shares the one array and it keeps the last call's contents.  The
// split partials are written before they are read within each call; the
// per-unit arrival counts are the one part that must start at zero, and each
// call clears them on its stream (one small cudaMemsetAsync) before its
// kernel.  So a call after a replay that timed out, or after a call of
// another context whose partials overlapped these counts, starts clean.
// Calls whose kernels overlap on the GPU (for example on two streams without
// ordering between them) race on the array.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fusedkv.h"
#include "fkv_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
// Device address of the array, per device, looked up once per process.  A
// device reset (cudaDeviceReset) ends the context that address belongs to;
// this library is not meant to outlive one, and after it these cached
// addresses would be stale.
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
fkv_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FKV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FKV_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FKV_OK;
}

}  // namespace

extern "C" {

fkv_status fkv_decode_attn_noalloc(fkv_ctx* ctx, const void* q, int layer, int mode,
                                   const int32_t* seq_lens, void* out, void* stream) {
  if (!ctx) return FKV_ERR_INVALID_ARG;
  if (fkv_decode_workspace_bytes(ctx) > kNoAllocScratchBytes) return FKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  const fkv_status s = scratch_for_current_device(&scratch);
  if (s != FKV_OK) return s;
  return fkv::decode_attn_impl(ctx, q, layer, mode, seq_lens, out, scratch,
                              kNoAllocScratchBytes, stream, /*clear_counts=*/true);
}

}  // extern "C"
