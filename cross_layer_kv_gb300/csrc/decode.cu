// Decode planning and dispatch by element type.
#include <algorithm>

#include "decode_impl.cuh"

namespace fkv {

cudaError_t decode_launch_bf16(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s);
cudaError_t decode_launch_f32(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s);
size_t decode_shape_bf16(int head_dim, int nsrc, int G, int B, int* warps);
size_t decode_shape_f32(int head_dim, int nsrc, int G, int B, int* warps);

// Rows (cache rows x KV heads) below which another warp does not pay off.
constexpr long long kMinRowsPerWarp = 64;

cudaError_t decode_plan(const DecodeArgs& a, int num_sms, DecodePlan* plan) {
  int W = 0;
  const size_t smem = a.is_f32 ? decode_shape_f32(a.head_dim, a.nsrc, a.group, a.batch, &W)
                               : decode_shape_bf16(a.head_dim, a.nsrc, a.group, a.batch, &W);
  if (smem == 0 || W == 0) return cudaErrorInvalidValue;
  // One CTA of W warps per SM (the stage rings take most of the shared
  // memory), capped so that every warp has a useful share of rows.
  const long long rows = (long long)a.batch * a.kv_heads * a.max_seq;
  long long ctas = a.num_ctas > 0 ? a.num_ctas : num_sms;
  const long long by_rows = (rows + kMinRowsPerWarp * W - 1) / (kMinRowsPerWarp * W);
  if (a.num_ctas <= 0) ctas = std::max(1LL, std::min(ctas, by_rows));
  plan->ctas = (int)ctas;
  plan->warps_per_cta = W;
  plan->smem_bytes = smem;
  const size_t units = (size_t)a.batch * a.kv_heads;
  const size_t slots = (size_t)ctas * W + units;
  plan->partial_bytes = (slots * a.group * partial_stride(a.head_dim) * sizeof(float) + 15) / 16 * 16;
  plan->workspace_bytes = plan->partial_bytes + units * sizeof(unsigned long long);
  return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  return a.is_f32 ? decode_launch_f32(a, plan, stream) : decode_launch_bf16(a, plan, stream);
}

}  // namespace fkv
