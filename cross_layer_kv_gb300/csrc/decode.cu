// Decode planning and dispatch by element type.
#include <algorithm>

#include "decode_impl.cuh"

namespace fkv {

cudaError_t decode_launch_bf16(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s);
cudaError_t decode_launch_f32(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s);
size_t decode_smem_bf16(int head_dim, int nsrc, int B);
size_t decode_smem_f32(int head_dim, int nsrc, int B);

// Rows (cache rows x KV heads) below which another warp does not pay off.
constexpr long long kMinRowsPerWarp = 64;

cudaError_t decode_plan(const DecodeArgs& a, int num_sms, DecodePlan* plan) {
  const size_t smem = a.is_f32 ? decode_smem_f32(a.head_dim, a.nsrc, a.batch)
                               : decode_smem_bf16(a.head_dim, a.nsrc, a.batch);
  if (smem == 0) return cudaErrorInvalidValue;
  // One CTA of kDecodeWarps warps per SM (the stage rings take most of the
  // shared memory), capped so that every warp has a useful share of rows.
  const long long rows = (long long)a.batch * a.kv_heads * a.max_seq;
  long long ctas = a.num_ctas > 0 ? a.num_ctas : num_sms;
  const long long by_rows = (rows + kMinRowsPerWarp * kDecodeWarps - 1) / (kMinRowsPerWarp * kDecodeWarps);
  if (a.num_ctas <= 0) ctas = std::max(1LL, std::min(ctas, by_rows));
  plan->ctas = (int)ctas;
  plan->warps_per_cta = kDecodeWarps;
  plan->smem_bytes = smem;
  const size_t slots = (size_t)ctas * kDecodeWarps + (size_t)a.batch * a.kv_heads;
  plan->workspace_bytes = slots * a.group * partial_stride(a.head_dim) * sizeof(float);
  return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  return a.is_f32 ? decode_launch_f32(a, plan, stream) : decode_launch_bf16(a, plan, stream);
}

}  // namespace fkv
