// Decode kernel instantiations for float caches (one translation unit per
// element type so they compile in parallel).
#include "decode_impl.cuh"

namespace fkv {

template <int D, int NSRC, bool WGT>
static cudaError_t by_group(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  switch (a.group) {
    case 1: return decode_launch_t<float, D, NSRC, WGT, 1>(a, pl, s);
    case 2: return decode_launch_t<float, D, NSRC, WGT, 2>(a, pl, s);
    case 4: return decode_launch_t<float, D, NSRC, WGT, 4>(a, pl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
static cudaError_t by_src(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  if (a.nsrc == 2) return by_group<D, 2, true>(a, pl, s);
  return a.a[0] ? by_group<D, 1, true>(a, pl, s) : by_group<D, 1, false>(a, pl, s);
}

cudaError_t decode_launch_f32(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  switch (a.head_dim) {
    case 64: return by_src<64>(a, pl, s);
    case 80: return by_src<80>(a, pl, s);
    case 96: return by_src<96>(a, pl, s);
    case 128: return by_src<128>(a, pl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, int NSRC>
static size_t shape_by_group(int G, int B, int* warps) {
  switch (G) {
    case 1: *warps = DecodeShape<float, D, NSRC, 1>::W; return decode_smem_bytes<float, D, NSRC, 1>(B);
    case 2: *warps = DecodeShape<float, D, NSRC, 2>::W; return decode_smem_bytes<float, D, NSRC, 2>(B);
    case 4: *warps = DecodeShape<float, D, NSRC, 4>::W; return decode_smem_bytes<float, D, NSRC, 4>(B);
    default: return 0;
  }
}

template <int D>
static size_t shape_by_src(int nsrc, int G, int B, int* warps) {
  return nsrc == 2 ? shape_by_group<D, 2>(G, B, warps) : shape_by_group<D, 1>(G, B, warps);
}

size_t decode_shape_f32(int head_dim, int nsrc, int G, int B, int* warps) {
  switch (head_dim) {
    case 64: return shape_by_src<64>(nsrc, G, B, warps);
    case 80: return shape_by_src<80>(nsrc, G, B, warps);
    case 96: return shape_by_src<96>(nsrc, G, B, warps);
    case 128: return shape_by_src<128>(nsrc, G, B, warps);
    default: return 0;
  }
}

}  // namespace fkv
