// Decode kernel instantiations for __nv_bfloat16 caches (one translation unit per
// element type so they compile in parallel).
#include "decode_impl.cuh"

namespace fkv {

template <int D, int NSRC>
static cudaError_t by_group(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  switch (a.group) {
    case 1: return decode_launch_t<__nv_bfloat16, D, NSRC, 1>(a, pl, s);
    case 2: return decode_launch_t<__nv_bfloat16, D, NSRC, 2>(a, pl, s);
    case 4: return decode_launch_t<__nv_bfloat16, D, NSRC, 4>(a, pl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
static cudaError_t by_src(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  return a.nsrc == 2 ? by_group<D, 2>(a, pl, s) : by_group<D, 1>(a, pl, s);
}

cudaError_t decode_launch_bf16(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  switch (a.head_dim) {
    case 64: return by_src<64>(a, pl, s);
    case 80: return by_src<80>(a, pl, s);
    case 96: return by_src<96>(a, pl, s);
    case 128: return by_src<128>(a, pl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
static size_t smem_by_src(int nsrc, int B) {
  return nsrc == 2 ? decode_smem_bytes<__nv_bfloat16, D, 2, 1>(B) : decode_smem_bytes<__nv_bfloat16, D, 1, 1>(B);
}

size_t decode_smem_bf16(int head_dim, int nsrc, int B) {
  switch (head_dim) {
    case 64: return smem_by_src<64>(nsrc, B);
    case 80: return smem_by_src<80>(nsrc, B);
    case 96: return smem_by_src<96>(nsrc, B);
    case 128: return smem_by_src<128>(nsrc, B);
    default: return 0;
  }
}

}  // namespace fkv
