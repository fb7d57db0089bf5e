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
    // a ring cache keeps position p + t at row (p + t) % ring
    const int rows = a.ring > 0 ? a.ring : a.max_seq;
    const int row = a.ring > 0 ? (p + t) % a.ring : p + t;
    const size_t dst = (((size_t)b * a.kv_heads + h) * rows + row) * chunks + c;
    reinterpret_cast<uint4*>(a.k_cache)[dst] = reinterpret_cast<const uint4*>(a.k_new)[src];
    reinterpret_cast<uint4*>(a.v_cache)[dst] = reinterpret_cast<const uint4*>(a.v_new)[src];
  }
}

// Quantising append for 4-bit layers: one thread per group of 16 channels of
// one new row.  min/max in fp32, scale = bf16((max - min) / 15) (IEEE
// division), code = clamp(rint((x - min) / scale), 0, 15) with the stored
// (bf16) scale; a constant group stores code 0.  Record layout per row:
// D/2 bytes of codes (channel 2i low nibble, 2i+1 high), then (scale, min)
// bf16 pairs per group, then zero padding to a multiple of 16 bytes.
__global__ void __launch_bounds__(256) append_q4_kernel(AppendArgs a) {
  grid_dep_trigger();
  grid_dep_wait();
  const int groups = a.head_dim / kQ4Group;
  const int rq = q4_row_bytes(a.head_dim);
  const long long per_seq = (long long)a.kv_heads * a.T * groups;
  const long long total = (long long)a.batch * per_seq;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * total;
       i += (long long)gridDim.x * blockDim.x) {
    const int which = i >= total;          // 0: K, 1: V
    const long long j = i - which * total;
    const int b = (int)(j / per_seq);
    long long r = j - (long long)b * per_seq;
    const int h = (int)(r / ((long long)a.T * groups));
    r -= (long long)h * a.T * groups;
    const int t = (int)(r / groups);
    const int g = (int)(r - (long long)t * groups);
    const int p = a.pos[b];
    if (p < 0 || (long long)p + a.T > a.max_seq) {
      if (h == 0 && t == 0 && g == 0 && which == 0) flag_status(a.status, kDevBadArg);
      continue;
    }
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(which ? a.v_new : a.k_new) +
                               ((((size_t)b * a.kv_heads + h) * a.T + t) * a.head_dim + g * kQ4Group);
    // a ring cache keeps position p + t at row (p + t) % ring
    const int rows = a.ring > 0 ? a.ring : a.max_seq;
    const int row = a.ring > 0 ? (p + t) % a.ring : p + t;
    uint8_t* rec = static_cast<uint8_t*>(which ? a.v_cache : a.k_cache) +
                   (((size_t)b * a.kv_heads + h) * rows + row) * rq;
    float x[kQ4Group];
    const uint4 w0 = reinterpret_cast<const uint4*>(src)[0];
    const uint4 w1 = reinterpret_cast<const uint4*>(src)[1];
    unpack16<__nv_bfloat16>(w0, x);
    unpack16<__nv_bfloat16>(w1, x + 8);
    float lo = x[0], hi = x[0];
#pragma unroll
    for (int e = 1; e < kQ4Group; ++e) {
      lo = fminf(lo, x[e]);
      hi = fmaxf(hi, x[e]);
    }
    const __nv_bfloat16 sb = __float2bfloat16_rn((hi - lo) / 15.0f);
    const float sc = __bfloat162float(sb);
    uint32_t code[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < kQ4Group; ++e) {
      float q = sc > 0.f ? rintf((x[e] - lo) / sc) : 0.f;
      q = fminf(fmaxf(q, 0.f), 15.f);
      code[e / 8] |= (uint32_t)q << (4 * (e % 8));
    }
    *reinterpret_cast<uint2*>(rec + g * 8) = make_uint2(code[0], code[1]);
    const __nv_bfloat16 lb = __float2bfloat16_rn(lo);
    const uint32_t prm = (uint32_t)__bfloat16_as_ushort(sb) | ((uint32_t)__bfloat16_as_ushort(lb) << 16);
    *reinterpret_cast<uint32_t*>(rec + a.head_dim / 2 + g * 4) = prm;
    if (g == 0) {
      for (int k = a.head_dim / 2 + a.head_dim / 4; k < rq; ++k) rec[k] = 0;
    }
  }
}

cudaError_t append_q4_launch(const AppendArgs& a, cudaStream_t stream) {
  const long long total = 2LL * a.batch * a.kv_heads * a.T * (a.head_dim / kQ4Group);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  return launch_pdl(append_q4_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

cudaError_t append_launch(const AppendArgs& a, cudaStream_t stream) {
  const long long total = (long long)a.batch * a.kv_heads * a.T * (a.head_dim * a.elem_bytes / 16);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  return launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

}  // namespace fkv
