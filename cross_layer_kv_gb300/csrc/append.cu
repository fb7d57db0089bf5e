// fkv_append_kv: write the post-RoPE K/V rows of T new tokens into a layer's
// cache at per-sequence positions (the storage caches take the new token
// before the upper layers attend; FusedKV reading notes §2.3).
//
// One thread moves 16 bytes; a row of D elements is D*e/16 threads, rows of
// the same (b, h) are contiguous on both sides, so reads and writes coalesce.
#include "fkv_device.cuh"
#include "fkv_kernels.h"

namespace fkv {

__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  grid_dep_trigger();
  grid_dep_wait();
  const int chunks = a.head_dim * a.elem_bytes / 16;   // 16-byte chunks per row
  const long long per_seq = (long long)a.kv_heads * a.T * chunks;
  const long long total = (long long)a.batch * per_seq;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / per_seq);
    long long r = i - (long long)b * per_seq;
    const int h = (int)(r / ((long long)a.T * chunks));
    r -= (long long)h * a.T * chunks;
    const int t = (int)(r / chunks);
    const int c = (int)(r - (long long)t * chunks);
    const int p = a.pos[b];
    if (p < 0 || (long long)p + a.T > a.max_seq) {
      if (h == 0 && t == 0 && c == 0) flag_status(a.status, kDevBadArg);
      continue;
    }
    const size_t src = (((size_t)b * a.kv_heads + h) * a.T + t) * chunks + c;
    const size_t dst = (((size_t)b * a.kv_heads + h) * a.max_seq + p + t) * chunks + c;
    reinterpret_cast<uint4*>(a.k_cache)[dst] = reinterpret_cast<const uint4*>(a.k_new)[src];
    reinterpret_cast<uint4*>(a.v_cache)[dst] = reinterpret_cast<const uint4*>(a.v_new)[src];
  }
}

cudaError_t append_launch(const AppendArgs& a, cudaStream_t stream) {
  const long long total = (long long)a.batch * a.kv_heads * a.T * (a.head_dim * a.elem_bytes / 16);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  return launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

}  // namespace fkv
