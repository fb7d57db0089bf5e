// The C ABI of include/fusedkv.h: context, host-side validation and dispatch
// to the kernels.  Every check runs before any launch; nothing here allocates
// on the hot path.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fusedkv.h"
#include "fkv_kernels.h"

struct fkv_ctx {
  fkv_config cfg;
  int n;          // storage layers 1..n
  int group;      // H_q / H_kv
  float scale;    // softmax scale
  int device;
  int num_sms;
  int* status;    // device words: the status (int32 at byte 0) and the
                  // limit of the bounded waits in ns (uint64 at byte 8)
  unsigned long long* wait_limit;
  std::vector<void*> k, v;                 // index: layer (1-based)
  std::vector<const float*> w[4];          // a_first, a_second, b_first, b_second
  std::vector<int> lite_src[2];            // lite / scaled sources: K, V
  std::vector<int> fused_src[4];           // fused sources: K first, K second, V first, V second
  std::vector<int> window;                 // sliding window per layer (0: full attention)
  std::vector<char> q4;                    // layer cache holds 4-bit records
  std::vector<int> ring;                   // > 0: the layer's caches are rings of that many rows
};

namespace {

// The device words of a context: status (int32) at byte 0, the limit of
// the bounded waits (uint64, ns) at byte 8.
constexpr size_t kDeviceWordsBytes = 16;
constexpr unsigned long long kDefaultWaitLimitNs = fkv::kWaitLimitNs;

// Process-wide call counter: tags each decode call's per-unit arrival counts
// so that counts left in a reused workspace by earlier calls never match.
std::atomic<unsigned> g_decode_epoch{1};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(const fkv_config& c) { return c.dtype == FKV_F32 ? 4 : 2; }

fkv_status check_config(const fkv_config* c) {
  if (!c) return FKV_ERR_INVALID_ARG;
  if (c->num_layers < 2 || c->num_layers % 2) return FKV_ERR_INVALID_ARG;
  if (c->batch < 1 || c->batch > 1024) return FKV_ERR_INVALID_ARG;
  if (c->max_seq < 1) return FKV_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->num_q_heads < 1) return FKV_ERR_INVALID_ARG;
  if (c->num_q_heads % c->num_kv_heads) return FKV_ERR_INVALID_ARG;
  if (c->dtype != FKV_BF16 && c->dtype != FKV_F32) return FKV_ERR_INVALID_ARG;
  if (!(c->softmax_scale >= 0.f) || !std::isfinite(c->softmax_scale)) return FKV_ERR_INVALID_ARG;
  if (c->decode_ctas < 0 || c->decode_ctas > 65535) return FKV_ERR_INVALID_ARG;
  if ((long long)c->batch * c->num_kv_heads * c->max_seq >= (1LL << 31)) return FKV_ERR_INVALID_ARG;
  const int g = c->num_q_heads / c->num_kv_heads;
  if (g != 1 && g != 2 && g != 4) return FKV_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 80 && c->head_dim != 96 && c->head_dim != 128)
    return FKV_ERR_UNSUPPORTED;
  return FKV_OK;
}

// Resolve the cache / weight sources of a call.  nsrc = 1 or 2.
fkv_status resolve_sources_impl(const fkv_ctx* c, int layer, int mode, const void* k[2],
                                const void* v[2], const float* a[2], const float* b[2], int* nsrc,
                                int src[4]) {
  if (layer < 1 || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  if (mode != FKV_VANILLA && mode != FKV_LITE && mode != FKV_FUSED && mode != FKV_SCALED)
    return FKV_ERR_INVALID_ARG;
  k[0] = k[1] = v[0] = v[1] = nullptr;
  a[0] = a[1] = b[0] = b[1] = nullptr;
  const int n = c->n;
  src[0] = src[1] = src[2] = src[3] = 0;
  if (layer <= n || mode == FKV_VANILLA) {
    if (layer > n && !c->cfg.store_upper) return FKV_ERR_UNSUPPORTED;
    k[0] = c->k[layer];
    v[0] = c->v[layer];
    src[0] = src[2] = layer;
    *nsrc = 1;
    if (!k[0] || !v[0]) return FKV_ERR_INVALID_ARG;
    return FKV_OK;
  }
  if (mode == FKV_LITE || mode == FKV_SCALED) {  // K^i = K^s, V^i = V^t (default n, 1)
    k[0] = c->k[c->lite_src[0][layer]];
    v[0] = c->v[c->lite_src[1][layer]];
    src[0] = c->lite_src[0][layer];
    src[2] = c->lite_src[1][layer];
    *nsrc = 1;
    if (!k[0] || !v[0]) return FKV_ERR_INVALID_ARG;
    if (mode == FKV_SCALED) {  // a_first scales K, b_first scales V
      a[0] = c->w[0][layer];
      b[0] = c->w[2][layer];
      if (!a[0] || !b[0]) return FKV_ERR_INVALID_ARG;
    }
    return FKV_OK;
  }
  // fused: K^s1, K^s2 with a_first, a_second; V^t1, V^t2 with b_first, b_second
  k[0] = c->k[c->fused_src[0][layer]];
  k[1] = c->k[c->fused_src[1][layer]];
  v[0] = c->v[c->fused_src[2][layer]];
  v[1] = c->v[c->fused_src[3][layer]];
  for (int i = 0; i < 4; ++i) src[i] = c->fused_src[i][layer];
  for (int i = 0; i < 2; ++i) {
    a[i] = c->w[i][layer];
    b[i] = c->w[2 + i][layer];
  }
  *nsrc = 2;
  if (!k[0] || !k[1] || !v[0] || !v[1] || !a[0] || !a[1] || !b[0] || !b[1])
    return FKV_ERR_INVALID_ARG;
  return FKV_OK;
}

// Sources and their storage format: *q4 = 1 if every source layer holds
// 4-bit records, 0 if none does; *ring = the row count of the sources' ring
// caches, 0 if they are full-length.  A mix of formats or of ring sizes is
// FKV_ERR_UNSUPPORTED (the sources of a call are read at the same rows).
fkv_status resolve_sources(const fkv_ctx* c, int layer, int mode, const void* k[2],
                           const void* v[2], const float* a[2], const float* b[2], int* nsrc,
                           int* q4, int* ring) {
  int src[4];
  const fkv_status s = resolve_sources_impl(c, layer, mode, k, v, a, b, nsrc, src);
  if (s != FKV_OK) return s;
  int nq = 0, nt = 0, r = -1;
  for (int i = 0; i < 4; ++i) {
    if (src[i] <= 0) continue;
    ++nt;
    nq += c->q4[src[i]] ? 1 : 0;
    if (r >= 0 && c->ring[src[i]] != r) return FKV_ERR_UNSUPPORTED;
    r = c->ring[src[i]];
  }
  if (nq != 0 && nq != nt) return FKV_ERR_UNSUPPORTED;
  *q4 = nq ? 1 : 0;
  *ring = r > 0 ? r : 0;
  return FKV_OK;
}

fkv::DecodeArgs decode_args(const fkv_ctx* c) {
  fkv::DecodeArgs d{};
  d.batch = c->cfg.batch;
  d.kv_heads = c->cfg.num_kv_heads;
  d.group = c->group;
  d.max_seq = c->cfg.max_seq;
  d.head_dim = c->cfg.head_dim;
  d.is_f32 = c->cfg.dtype == FKV_F32;
  d.softmax_scale = c->scale;
  d.status = c->status;
  d.wait_limit = c->wait_limit;
  d.num_ctas = c->cfg.decode_ctas;
  return d;
}

}  // namespace

namespace fkv {

// One decode call after host validation (see fkv_decode_attn).  With
// clear_counts the unit arrival words of this call's plan are zeroed on the
// stream before the launch (the no-allocation entry point, whose caller
// cannot reach its scratch array to clear it after a timed-out replay).
fkv_status decode_attn_impl(fkv_ctx* c, const void* q, int layer, int mode,
                            const int32_t* seq_lens, void* out, void* workspace,
                            size_t workspace_bytes, void* stream, bool clear_counts) {
  if (!c) return FKV_ERR_INVALID_ARG;
  fkv::DecodeArgs d = decode_args(c);
  int q4 = 0, ring = 0;
  fkv_status s = resolve_sources(c, layer, mode, d.k, d.v, d.a, d.b, &d.nsrc, &q4, &ring);
  if (s != FKV_OK) return s;
  // ring caches hold the last `ring` positions: the layer must attend within them
  if (ring > 0 && (c->window[layer] < 1 || c->window[layer] > ring)) return FKV_ERR_INVALID_ARG;
  if (!q || !out || !seq_lens || !aligned16(q) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return FKV_ERR_INVALID_ARG;
  fkv::DecodePlan plan{};
  const cudaError_t pe = q4 ? fkv::decode_q4_plan(d, c->num_sms, &plan)
                            : fkv::decode_plan(d, c->num_sms, &plan);
  if (pe != cudaSuccess) return FKV_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < plan.workspace_bytes)
    return FKV_ERR_WORKSPACE;
  d.q = q;
  d.out = out;
  d.seq_lens = seq_lens;
  d.workspace = static_cast<float*>(workspace);
  d.window = c->window[layer];
  d.ring = ring;
  unsigned ep = g_decode_epoch.fetch_add(1);
  if (ep == 0) ep = g_decode_epoch.fetch_add(1);
  d.epoch = ep;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clear_counts &&
      cudaMemsetAsync(static_cast<char*>(workspace) + plan.partial_bytes, 0,
                      plan.workspace_bytes - plan.partial_bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return FKV_ERR_CUDA;
  }
  const cudaError_t e = q4 ? fkv::decode_q4_launch(d, plan, st) : fkv::decode_launch(d, plan, st);
  return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

}  // namespace fkv

extern "C" {

fkv_status fkv_create(const fkv_config* cfg, fkv_ctx** out) {
  if (!out) return FKV_ERR_INVALID_ARG;
  *out = nullptr;
  fkv_status s = check_config(cfg);
  if (s != FKV_OK) return s;
  fkv_ctx* c = new (std::nothrow) fkv_ctx();
  if (!c) return FKV_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->n = cfg->num_layers / 2;
  c->group = cfg->num_q_heads / cfg->num_kv_heads;
  c->scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / std::sqrt((float)cfg->head_dim);
  c->k.assign(cfg->num_layers + 1, nullptr);
  c->v.assign(cfg->num_layers + 1, nullptr);
  for (auto& w : c->w) w.assign(cfg->num_layers + 1, nullptr);
  c->window.assign(cfg->num_layers + 1, 0);
  c->q4.assign(cfg->num_layers + 1, 0);
  c->ring.assign(cfg->num_layers + 1, 0);
  c->lite_src[0].assign(cfg->num_layers + 1, c->n);  // K^n
  c->lite_src[1].assign(cfg->num_layers + 1, 1);     // V^1
  c->fused_src[0].assign(cfg->num_layers + 1, 1);
  c->fused_src[1].assign(cfg->num_layers + 1, c->n);
  c->fused_src[2].assign(cfg->num_layers + 1, 1);
  c->fused_src[3].assign(cfg->num_layers + 1, c->n);
  c->status = nullptr;
  c->wait_limit = nullptr;
  const unsigned long long limit = kDefaultWaitLimitNs;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess ||
      cudaMalloc(&c->status, kDeviceWordsBytes) != cudaSuccess ||
      cudaMemset(c->status, 0, kDeviceWordsBytes) != cudaSuccess ||
      cudaMemcpy(reinterpret_cast<char*>(c->status) + 8, &limit, sizeof(limit),
                 cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    if (c->status) cudaFree(c->status);
    delete c;
    return FKV_ERR_CUDA;
  }
  c->wait_limit = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(c->status) + 8);
  *out = c;
  return FKV_OK;
}

void fkv_destroy(fkv_ctx* c) {
  if (!c) return;
  if (c->status) cudaFree(c->status);
  delete c;
}

fkv_status fkv_bind_layer_cache(fkv_ctx* c, int layer, void* k, void* v) {
  if (!c || layer < 1 || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  if (layer > c->n && !c->cfg.store_upper) return FKV_ERR_UNSUPPORTED;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return FKV_ERR_INVALID_ARG;
  c->k[layer] = k;
  c->v[layer] = v;
  c->q4[layer] = 0;
  return FKV_OK;
}

size_t fkv_q4_row_bytes(int head_dim) {
  if (head_dim != 64 && head_dim != 80 && head_dim != 96 && head_dim != 128) return 0;
  return (size_t)fkv::q4_row_bytes(head_dim);
}

fkv_status fkv_bind_layer_cache_q4(fkv_ctx* c, int layer, void* k_rec, void* v_rec) {
  if (!c || layer < 1 || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  if (c->cfg.dtype != FKV_BF16 || c->group > 2) return FKV_ERR_UNSUPPORTED;
  if (layer > c->n && !c->cfg.store_upper) return FKV_ERR_UNSUPPORTED;
  if (!k_rec || !v_rec || !aligned16(k_rec) || !aligned16(v_rec)) return FKV_ERR_INVALID_ARG;
  c->k[layer] = k_rec;
  c->v[layer] = v_rec;
  c->q4[layer] = 1;
  return FKV_OK;
}

fkv_status fkv_set_fusion_weights(fkv_ctx* c, int layer, const float* a_first,
                                  const float* a_second, const float* b_first,
                                  const float* b_second) {
  if (!c || layer <= c->n || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  const float* ws[4] = {a_first, a_second, b_first, b_second};
  for (int i = 0; i < 4; ++i)
    if (!ws[i] || !aligned16(ws[i])) return FKV_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) c->w[i][layer] = ws[i];
  return FKV_OK;
}

fkv_status fkv_set_sources(fkv_ctx* c, int layer, int mode, int k_first, int k_second,
                           int v_first, int v_second) {
  if (!c || layer <= c->n || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  auto storage = [&](int l) { return l >= 1 && l <= c->n; };
  if (mode == FKV_LITE || mode == FKV_SCALED) {
    if (!storage(k_first) || !storage(v_first)) return FKV_ERR_INVALID_ARG;
    c->lite_src[0][layer] = k_first;
    c->lite_src[1][layer] = v_first;
    return FKV_OK;
  }
  if (mode == FKV_FUSED) {
    if (!storage(k_first) || !storage(k_second) || !storage(v_first) || !storage(v_second))
      return FKV_ERR_INVALID_ARG;
    c->fused_src[0][layer] = k_first;
    c->fused_src[1][layer] = k_second;
    c->fused_src[2][layer] = v_first;
    c->fused_src[3][layer] = v_second;
    return FKV_OK;
  }
  return FKV_ERR_INVALID_ARG;
}

fkv_status fkv_set_window(fkv_ctx* c, int layer, int window) {
  if (!c || layer < 1 || layer > c->cfg.num_layers || window < 0) return FKV_ERR_INVALID_ARG;
  c->window[layer] = window;
  return FKV_OK;
}

fkv_status fkv_set_ring_rows(fkv_ctx* c, int layer, int rows) {
  if (!c || layer < 1 || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  if (rows < 0 || rows > c->cfg.max_seq) return FKV_ERR_INVALID_ARG;
  c->ring[layer] = rows == c->cfg.max_seq ? 0 : rows;
  return FKV_OK;
}

fkv_status fkv_append_kv(fkv_ctx* c, int layer, const void* k_new, const void* v_new,
                         const int32_t* pos, int T, void* stream) {
  if (!c || layer < 1 || layer > c->cfg.num_layers) return FKV_ERR_INVALID_ARG;
  if (layer > c->n && !c->cfg.store_upper) return FKV_ERR_UNSUPPORTED;
  if (T < 0 || T > c->cfg.max_seq) return FKV_ERR_INVALID_ARG;
  if (c->ring[layer] > 0 && T > c->ring[layer]) return FKV_ERR_INVALID_ARG;
  if (!c->k[layer] || !c->v[layer]) return FKV_ERR_INVALID_ARG;
  if (T == 0) return FKV_OK;
  if (!k_new || !v_new || !pos || !aligned16(k_new) || !aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return FKV_ERR_INVALID_ARG;
  fkv::AppendArgs a{};
  a.k_cache = c->k[layer];
  a.v_cache = c->v[layer];
  a.k_new = k_new;
  a.v_new = v_new;
  a.pos = pos;
  a.status = c->status;
  a.batch = c->cfg.batch;
  a.kv_heads = c->cfg.num_kv_heads;
  a.max_seq = c->cfg.max_seq;
  a.head_dim = c->cfg.head_dim;
  a.T = T;
  a.elem_bytes = elem_bytes(c->cfg);
  a.ring = c->ring[layer];
  const cudaError_t e = c->q4[layer] ? fkv::append_q4_launch(a, static_cast<cudaStream_t>(stream))
                                     : fkv::append_launch(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

size_t fkv_decode_workspace_bytes(const fkv_ctx* c) {
  if (!c) return 0;
  size_t best = 0;
  for (int nsrc = 1; nsrc <= 2; ++nsrc) {
    fkv::DecodeArgs d = decode_args(c);
    d.nsrc = nsrc;
    fkv::DecodePlan p{};
    if (fkv::decode_plan(d, c->num_sms, &p) == cudaSuccess && p.workspace_bytes > best)
      best = p.workspace_bytes;
    if (fkv::decode_q4_plan(d, c->num_sms, &p) == cudaSuccess && p.workspace_bytes > best)
      best = p.workspace_bytes;
  }
  return best;
}

fkv_status fkv_decode_attn(fkv_ctx* c, const void* q, int layer, int mode,
                           const int32_t* seq_lens, void* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return fkv::decode_attn_impl(c, q, layer, mode, seq_lens, out, workspace, workspace_bytes,
                               stream, false);
}

fkv_status fkv_prefill_attn(fkv_ctx* c, const void* q, int layer, int mode, int S, void* out,
                            void* stream) {
  return fkv_prefill_attn_chunk(c, q, layer, mode, 0, S, out, stream);
}

fkv_status fkv_prefill_attn_chunk(fkv_ctx* c, const void* q, int layer, int mode, int q_start,
                                  int C, void* out, void* stream) {
  if (!c) return FKV_ERR_INVALID_ARG;
  const int S = C;
  fkv::PrefillArgs p{};
  int q4 = 0, ring = 0;
  fkv_status s = resolve_sources(c, layer, mode, p.k, p.v, p.a, p.b, &p.nsrc, &q4, &ring);
  if (s != FKV_OK) return s;
  if (q4) return FKV_ERR_UNSUPPORTED;   // prefill reads bf16 caches
  if (c->cfg.dtype != FKV_BF16) return FKV_ERR_UNSUPPORTED;
  if (S < 1 || q_start < 0 || (long long)q_start + S > c->cfg.max_seq) return FKV_ERR_INVALID_ARG;
  // Over ring caches whose positions have wrapped, every key a query of the
  // chunk attends must still be in the ring: a sliding window W with
  // C + W - 1 <= rows (the kernels also want rows to be a multiple of their
  // key tile, else FKV_ERR_UNSUPPORTED).
  if (ring > 0 && (long long)q_start + S > ring) {
    const int W = c->window[layer];
    if (W < 1 || W > ring) return FKV_ERR_INVALID_ARG;
    if ((long long)S + W - 1 > ring) return FKV_ERR_UNSUPPORTED;
  }
  p.plane_rows = ring > 0 ? ring : c->cfg.max_seq;
  p.ring = ring;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return FKV_ERR_INVALID_ARG;
  p.q_start = q_start;
  p.window = c->window[layer];
  p.q = q;
  p.out = out;
  p.status = c->status;
  p.wait_limit = c->wait_limit;
  p.batch = c->cfg.batch;
  p.kv_heads = c->cfg.num_kv_heads;
  p.group = c->group;
  p.max_seq = c->cfg.max_seq;
  p.head_dim = c->cfg.head_dim;
  p.S = S;
  p.softmax_scale = c->scale;
  const cudaError_t e = fkv::prefill_launch(p, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return FKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FKV_OK : FKV_ERR_CUDA;
}

fkv_status fkv_get_device_status(fkv_ctx* c, void* stream) {
  if (!c) return FKV_ERR_INVALID_ARG;
  int h = 0;
  if (cudaMemcpyAsync(&h, c->status, sizeof(int), cudaMemcpyDeviceToHost,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FKV_ERR_CUDA;
  }
  if (h == 0) return FKV_OK;
  if (cudaMemsetAsync(c->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FKV_ERR_CUDA;
  return (h & fkv::kDevTimeoutBit) ? FKV_ERR_TIMEOUT : FKV_ERR_DEVICE_ARG;
}

fkv_status fkv_set_wait_limit(fkv_ctx* c, unsigned long long limit_ns) {
  if (!c) return FKV_ERR_INVALID_ARG;
  if (limit_ns > kDefaultWaitLimitNs) return FKV_ERR_INVALID_ARG;
  if (cudaMemcpy(c->wait_limit, &limit_ns, sizeof(limit_ns), cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaGetLastError();
    return FKV_ERR_CUDA;
  }
  return FKV_OK;
}

const char* fkv_status_string(fkv_status s) {
  switch (s) {
    case FKV_OK: return "ok";
    case FKV_ERR_INVALID_ARG: return "invalid argument";
    case FKV_ERR_UNSUPPORTED: return "unsupported";
    case FKV_ERR_CUDA: return "CUDA error";
    case FKV_ERR_TIMEOUT: return "device wait timed out";
    case FKV_ERR_WORKSPACE: return "workspace missing or too small";
    case FKV_ERR_DEVICE_ARG: return "device saw an out-of-range length or position";
  }
  return "unknown status";
}

}  // extern "C"
