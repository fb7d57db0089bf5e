// Host-visible launch interfaces of the FusedKV kernels (internal to the
// library; the public ABI is include/fusedkv.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fusedkv.h"

namespace fkv {

// Default limit of every bounded device wait (a context's wait-limit word
// starts here; only the failure-path tests lower it).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// One decode attention call, after host validation.  Pointers are device
// pointers.  nsrc = 1: K from k[0], V from v[0] (vanilla or lite);
// nsrc = 2: fused, K = a0 (.) k[0] + a1 (.) k[1], V = b0 (.) v[0] + b1 (.) v[1].
struct DecodeArgs {
  const void* k[2];
  const void* v[2];
  const float* a[2];
  const float* b[2];
  const void* q;             // [B, H_q, D]
  void* out;                 // [B, H_q, D]
  const int32_t* seq_lens;   // [B]
  float* workspace;          // split partials
  int* status;               // device status word
  const unsigned long long* wait_limit;  // device word: limit of the bounded waits (ns)
  int batch, kv_heads, group, max_seq, head_dim;
  int nsrc;
  int is_f32;
  float softmax_scale;
  int num_ctas;              // split grid (0 = library default)
  int window;                // > 0: attend only to the last `window` rows
  int ring;                  // > 0: the source caches are rings of this many rows per
                             // unit (position t at row t % ring); 0: S_max rows, row = position
  unsigned epoch;            // distinct per call (tags the unit arrival counts)
};

// Launch configuration the library picks for a decode call shape.
struct DecodePlan {
  int ctas;          // CTAs of the split kernel
  int warps_per_cta;
  size_t smem_bytes;
  size_t partial_bytes;    // split partials, then one 8-byte arrival word per unit
  size_t workspace_bytes;
};

// Plan (grid and workspace) for a shape; num_sms from the device.
cudaError_t decode_plan(const DecodeArgs& a, int num_sms, DecodePlan* plan);

// Launch the decode kernel on `stream`.
cudaError_t decode_launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);

// Number of kernel launches one decode call makes (for launch accounting).
constexpr int kDecodeLaunchesPerCall = 1;

// Launch `kern` with programmatic stream serialization (see grid_dep_wait).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct AppendArgs {
  void* k_cache;
  void* v_cache;
  const void* k_new;
  const void* v_new;
  const int32_t* pos;
  int* status;
  int batch, kv_heads, max_seq, head_dim, T, elem_bytes;
  int ring;        // > 0: the cache is a ring of this many rows per unit (row = position % ring)
};

cudaError_t append_launch(const AppendArgs& a, cudaStream_t stream);

// 4-bit caches: rows of q4_row_bytes(D) bytes (codes, then bf16 (scale, min)
// per group of kQ4Group channels, padded to 16 bytes).
constexpr int kQ4Group = 16;
__host__ __device__ constexpr int q4_row_bytes(int head_dim) {
  return (head_dim / 2 + head_dim / 4 + 15) / 16 * 16;
}
cudaError_t append_q4_launch(const AppendArgs& a, cudaStream_t stream);
cudaError_t decode_q4_launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);
cudaError_t decode_q4_plan(const DecodeArgs& a, int num_sms, DecodePlan* plan);

constexpr int kDevTimeoutBit = 2;  // must match kDevTimeout

struct PrefillArgs {
  const void* k[2];
  const void* v[2];
  const float* a[2];
  const float* b[2];
  const void* q;   // [B, H_q, S, D] bf16
  void* out;       // [B, H_q, S, D] bf16
  int* status;
  const unsigned long long* wait_limit;  // device word: limit of the bounded waits (ns)
  int batch, kv_heads, group, max_seq, head_dim, S;
  int q_start;     // cache position of query row 0 (0 for a whole prompt)
  int window;      // > 0: sliding window of that many positions
  int plane_rows;  // cache rows per (b, kv-head) unit (S_max, or a ring's rows)
  int ring;        // > 0: the caches are rings of that many rows (position t at row
                   // t % ring), a multiple of the kernel's key tile once positions wrap
  int nsrc;
  float softmax_scale;
};

// Returns cudaErrorNotSupported for shapes the tensor-core kernels do not
// cover.  One source (nsrc = 1) runs the 128-key kernel of prefill_wide.cu;
// two sources (fused) with D <= 96 the 112-key kernel of
// prefill_fused_wide.cu (Q in tensor memory), and with D = 128 the 64-key
// kernel of prefill.cu.
cudaError_t prefill_launch(const PrefillArgs& a, cudaStream_t stream);
cudaError_t prefill_wide_launch(const PrefillArgs& a, cudaStream_t stream);
cudaError_t prefill_fused_wide_launch(const PrefillArgs& a, cudaStream_t stream);

// The body of fkv_decode_attn (api.cu); clear_counts zeroes the call's unit
// arrival words on the stream before the launch.  Internal to the library.
__attribute__((visibility("hidden"))) fkv_status decode_attn_impl(
    fkv_ctx* c, const void* q, int layer, int mode, const int32_t* seq_lens, void* out,
    void* workspace, size_t workspace_bytes, void* stream, bool clear_counts);

}  // namespace fkv
