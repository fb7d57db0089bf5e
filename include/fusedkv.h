/*
 * fusedkv.h -- C ABI of the FusedKV attention library for GB300 (sm_103a).
 *
 * FusedKV ("Reconstructing KV Caches with Cross-Layer Fusion for Enhanced
 * Transformers", Lin et al., arXiv:2512.03870) keeps post-RoPE K/V caches only
 * for the lower half of the layers.  With L = 2n layers (1-based):
 *
 *   storage layers        1..n    attend over their own stored K/V;
 *   reconstruction layers n+1..L  rebuild K/V on demand from layers 1 and n:
 *     fused (FusedKV slides, Eqs.(4)-(5)):
 *        K^i = a_{i,1} (.) K^1 + a_{i,n} (.) K^n
 *        V^i = b_{i,1} (.) V^1 + b_{i,n} (.) V^n
 *     lite  (FusedKV slides, Eq.(6)):  K^i = K^n,  V^i = V^1
 *     vanilla (Table 1, the full-cache baseline): every layer stores its own.
 *
 * The reconstruction happens inside the attention kernels; reconstructed upper
 * layer K/V is never written to memory (FusedKV slides, Table 1 slide: "fuse on
 * demand"; reading notes §2.3).
 *
 * Conventions used by every call:
 *   - Layers are 1-based, L even, n = L / 2 (reading notes §2.1, Eq.(1)).
 *   - Caches are caller-owned device buffers, contiguous [B, H_kv, S_max, D],
 *     holding post-RoPE keys and values; element type = the context dtype.
 *   - Fusion weights are caller-owned device fp32 buffers [H_kv, D] per
 *     target layer (one weight per KV head and channel, broadcast over batch
 *     and tokens).  The key weights should be tied across each RoPE rotation
 *     pair (channel j with j + D/2 in rotate-half storage; FusedKV slides,
 *     Eqs.(7)-(8)); the library does not enforce it.
 *   - GQA: query head h reads KV head h / (H_q / H_kv).
 *   - Softmax scale: config.softmax_scale, or 1/sqrt(D) when it is 0.
 *   - Device pointers must be 16-byte aligned.
 *   - Every call is asynchronous and ordered on the given stream (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - Host-side validation happens before any launch; a failing call
 *     launches nothing.  Conditions only the device can see (a sequence
 *     length out of range, a bounded wait that ran out) are recorded in a
 *     device status word read by fkv_get_device_status().
 *   - Nothing aborts, throws or allocates on the hot path; the library owns
 *     only its context (and, after fkv_create, 16 bytes of device words: the
 *     status word and the limit of the bounded waits).
 */
#ifndef FUSEDKV_H_
#define FUSEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FKV_OK = 0,
  FKV_ERR_INVALID_ARG = 1,  /* bad pointer, size, layer, alignment or config */
  FKV_ERR_UNSUPPORTED = 2,  /* valid request this library or config cannot serve */
  FKV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  FKV_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out */
  FKV_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
  FKV_ERR_DEVICE_ARG = 6    /* device saw a sequence length / position out of range */
} fkv_status;

typedef enum {
  FKV_VANILLA = 0, /* the layer's own cache (Table 1's full-cache baseline) */
  FKV_LITE = 1,    /* K^i = K^s, V^i = V^t; (s, t) = (n, 1) unless set (Eq.(6)) */
  FKV_FUSED = 2,   /* K^i = a1 (.) K^s1 + a2 (.) K^s2, likewise V; (1, n) unless set (Eqs.(4)-(5)) */
  FKV_SCALED = 3   /* K^i = a1 (.) K^s, V^i = b1 (.) V^t on the Lite sources: the
                      single-source learnable channel scaling of the FusedKV
                      slides' Fig.8 ablation */
} fkv_mode;

typedef enum { FKV_BF16 = 0, FKV_F32 = 1 } fkv_dtype;

typedef struct {
  int num_layers;     /* L, even, >= 2 */
  int batch;          /* B, 1..1024 */
  int max_seq;        /* S_max: cache rows per (batch, KV head) */
  int num_q_heads;    /* H_q, a multiple of H_kv, H_q / H_kv in {1, 2, 4} */
  int num_kv_heads;   /* H_kv */
  int head_dim;       /* D in {64, 80, 96, 128} */
  int dtype;          /* fkv_dtype of caches, queries and outputs */
  int store_upper;    /* 1: upper layers also keep their own caches, so that
                         vanilla attention can run on them (comparison path) */
  float softmax_scale;/* 0 => 1/sqrt(D) */
  int decode_ctas;    /* 0: the library picks the decode split grid (one CTA
                         per SM, fewer for short caches); > 0 forces that
                         many CTAs (results agree up to fp32 rounding) */
} fkv_config;

typedef struct fkv_ctx fkv_ctx;

/* Create a context for the current CUDA device.  Validates the config
 * (FKV_ERR_INVALID_ARG / FKV_ERR_UNSUPPORTED before touching CUDA), then
 * queries the device and allocates its 16 bytes of device words, the status
 * word and the wait limit (FKV_ERR_CUDA on failure, e.g. no GPU).  *out is
 * set to NULL on any error. */
fkv_status fkv_create(const fkv_config* cfg, fkv_ctx** out);

/* Free the context and its device words.  NULL is ignored.  Does not touch
 * caller buffers. */
void fkv_destroy(fkv_ctx* ctx);

/* Register the K and V cache buffers of a layer (device, [B,H_kv,S_max,D],
 * 16-byte aligned).  Storage layers 1..n always have caches; upper layers only
 * when config.store_upper is set (else FKV_ERR_UNSUPPORTED: upper layers store
 * nothing, reading notes §2.1).  The buffers stay owned by the caller and must
 * outlive their use. */
fkv_status fkv_bind_layer_cache(fkv_ctx* ctx, int layer, void* k, void* v);

/* Bytes of one row of a 4-bit cache for head dim D (0 if D is unsupported):
 * D/2 bytes of codes, D/4 bytes of parameters, padded to 16 bytes
 * (48, 64, 80, 96 for D = 64, 80, 96, 128). */
size_t fkv_q4_row_bytes(int head_dim);

/* Register 4-bit K and V caches of a layer (FusedKV slides, "Four-bit KV
 * quantization is the stronger combination", Table 14; the quantisation
 * grouping is this library's, the pages do not give KIVI's):
 * k_rec, v_rec: device, [B, H_kv, S_max, fkv_q4_row_bytes(D)] bytes,
 * 16-byte aligned.  Each row holds its D channels in groups of 16 as 4-bit
 * codes (byte i: channel 2i in the low nibble, 2i+1 in the high one),
 * followed by one (scale, min) bf16 pair per group: x = min + code * scale.
 * fkv_append_kv quantises new rows of such a layer (min/max of the group,
 * scale = bf16((max - min) / 15), code = clamp(rint((x - min) / scale),
 * 0, 15)); fkv_decode_attn reads, dequantises and fuses them in registers when
 * every source layer of the call is 4-bit (a mix of formats, and prefill, give
 * FKV_ERR_UNSUPPORTED).  Needs dtype FKV_BF16 and H_q / H_kv <= 2. */
fkv_status fkv_bind_layer_cache_q4(fkv_ctx* ctx, int layer, void* k_rec, void* v_rec);

/* Register the fusion weights of reconstruction layer n < layer <= L
 * (FusedKV slides, Eqs.(4)-(5)): a_first/a_second scale K^1/K^n, b_first/
 * b_second scale V^1/V^n.  Each is a device fp32 [H_kv, D] buffer owned by the
 * caller.  Any sign and any sum are allowed. */
fkv_status fkv_set_fusion_weights(fkv_ctx* ctx, int layer, const float* a_first,
                                  const float* a_second, const float* b_first,
                                  const float* b_second);

/* Choose the stored layers an upper layer n < layer <= L reconstructs from
 * (FusedKV slides, "source-layer choice", Table 17, and the reversed sharing
 * K^1, V^n of Fig.8).  For mode FKV_LITE or FKV_SCALED, K comes from layer
 * k_first and V from layer v_first (k_second and v_second are ignored); for
 * FKV_FUSED, K from layers k_first and k_second (weighted by a_first,
 * a_second) and V from v_first and v_second (b_first, b_second).  Every
 * source must be a storage layer 1..n.  Defaults: Lite / scaled (n, 1),
 * fused (1, n, 1, n).  The caches must be bound before a call reads them. */
fkv_status fkv_set_sources(fkv_ctx* ctx, int layer, int mode, int k_first, int k_second,
                           int v_first, int v_second);

/* Make `layer` a sliding-window layer: its decode and prefill calls attend
 * only to the last `window` positions (keys t with m - window < t <= m for a
 * query at position m); 0 restores full attention (the default).  This is the
 * hybrid sliding-window setting of the FusedKV slides ("MoE and hybrid SWA":
 * window 512, three window layers per full-attention layer).  With
 * fkv_set_sources, window upper layers reconstruct from window storage layers
 * and full layers from full ones (sources typed by attention kind).  The
 * caches keep their [B, H_kv, S_max, D] layout; a window layer reads only
 * rows [len - window, len).  FKV_ERR_INVALID_ARG for a bad layer or a
 * negative window. */
fkv_status fkv_set_window(fkv_ctx* ctx, int layer, int window);

/* Make the caches of `layer` rings of `rows` rows per (batch row, KV head):
 * position t of a sequence lives at row t % rows, so a sliding-window layer
 * stores only the positions its window can reach instead of S_max rows (the
 * capacity half of the hybrid sliding-window sharing of the FusedKV slides,
 * "MoE and hybrid SWA").  The buffers bound to the layer (fkv_bind_layer_cache
 * or fkv_bind_layer_cache_q4, before or after this call) are then
 * [B, H_kv, rows, D] (or rows records).  rows = 0 (or S_max) restores the
 * full-length layout; FKV_ERR_INVALID_ARG for a bad layer or rows outside
 * [0, S_max].
 * Calls over ring caches:
 *   - fkv_append_kv writes position pos[b] + i at row (pos[b] + i) % rows;
 *     T <= rows (FKV_ERR_INVALID_ARG otherwise); rows of positions older than
 *     the last `rows` are overwritten, so append every position in order;
 *   - fkv_decode_attn needs every source of the call to be a ring of the same
 *     size (FKV_ERR_UNSUPPORTED otherwise) and the attending layer to have a
 *     window with 1 <= window <= rows (FKV_ERR_INVALID_ARG otherwise); a tile
 *     of rows that wraps past the ring's end is read in two copies;
 *   - fkv_prefill_attn / _chunk read rows as they are while the call's
 *     positions have not wrapped (q_start + C <= rows).  Past that, the layer
 *     needs a window 1 <= W <= rows (FKV_ERR_INVALID_ARG otherwise), the chunk
 *     C + W - 1 <= rows, and rows a multiple of the kernel's key tile: 128
 *     for one source, 112 for fused layers with head_dim <= 96, 64 for fused
 *     layers with head_dim 128 (FKV_ERR_UNSUPPORTED otherwise; 896 suits all
 *     three).  Every row must then have been written once, since rows past
 *     the chunk's last position are read and masked. */
fkv_status fkv_set_ring_rows(fkv_ctx* ctx, int layer, int rows);

/* Write the post-RoPE K/V of T new tokens into a layer's cache (the storage
 * caches take the new token before the upper layers attend; reading notes
 * §2.3).  k_new, v_new: device [B, H_kv, T, D] in the context dtype.
 * pos: device int32 [B], first cache row to write for each sequence.
 * Rows pos[b]..pos[b]+T-1 of every KV head are written; a sequence whose rows
 * fall outside [0, S_max) is skipped and flagged as FKV_ERR_DEVICE_ARG in the
 * device status.  The layer must have a bound cache. */
fkv_status fkv_append_kv(fkv_ctx* ctx, int layer, const void* k_new, const void* v_new,
                         const int32_t* pos, int T, void* stream);

/* Bytes of device workspace fkv_decode_attn needs for this context (split-K
 * partial results).  The caller allocates it; its contents need no
 * initialisation and may be reused by every decode call on the same stream. */
size_t fkv_decode_workspace_bytes(const fkv_ctx* ctx);

/* One decode attention call of a layer (a single query position per sequence).
 * What it computes: softmax attention of each query head over the layer's
 * keys and values, where an upper layer's K/V are those of FusedKV slides
 * "FusedKV learns two-source, channel-wise fusion", Eqs.(4)-(5) (fused) or
 * "Lite separates the key source from the value source", Eq.(6) (lite),
 * rebuilt on demand inside the kernel and never stored ("Half the storage can
 * require 50% more cache I/O", Table 1: fused reads K^1, K^n, V^1, V^n, twice
 * the bytes of a vanilla or lite call; reading notes §2.5 explains why decode
 * can therefore be slower while storage halves).
 * q: device [B, H_q, D]; out: device [B, H_q, D]; both in the context dtype.
 * seq_lens: device int32 [B]; sequence b attends over cache rows
 * [0, seq_lens[b]) (the new token already appended).  A length outside
 * [1, S_max] is clamped (0 yields a zero output) and flagged as
 * FKV_ERR_DEVICE_ARG in the device status.
 * mode: for storage layers every mode is plain attention over the layer's own
 * cache; for upper layers FKV_VANILLA reads the layer's own cache (needs
 * store_upper), FKV_LITE reads K^n and V^1, FKV_FUSED reads K^1, K^n, V^1, V^n
 * with the layer's weights and fuses them in registers, FKV_SCALED reads K^n
 * and V^1 scaled by a_first and b_first (sources as set by fkv_set_sources).
 * workspace: device, at least fkv_decode_workspace_bytes(ctx) bytes.
 * The call launches one kernel on `stream` and makes no synchronising CUDA
 * call, so it can be captured into a CUDA graph.  Every replay computes
 * afresh: the kernel clears the arrival counts it used once it is done.  A
 * replay that stopped early (FKV_ERR_TIMEOUT in the device status) can leave
 * counts behind under the captured call's tag; zero the workspace before the
 * next replay (a zero word is never a live count). */
fkv_status fkv_decode_attn(fkv_ctx* ctx, const void* q, int layer, int mode,
                           const int32_t* seq_lens, void* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/* fkv_decode_attn without a caller workspace.  The paper has no counterpart:
 * this is a deployment convenience of this library.
 *
 * It serves callers that cannot allocate device memory: a host process whose
 * device memory is fully reserved by its own pool allocator, or a plugin
 * interface that passes only the operands of one operation.  cudaMalloc is no
 * way out for them, since it synchronises the device and fails once memory is
 * exhausted.  This call runs the same kernels as fkv_decode_attn, with the
 * split partials in a 4 MiB array that the library holds in static device
 * memory on every GPU that loads it, until the process exits.  It calls no
 * allocator.
 *
 * Arguments and results are those of fkv_decode_attn without workspace and
 * workspace_bytes.  A context whose fkv_decode_workspace_bytes() exceeds
 * 4 MiB gets FKV_ERR_WORKSPACE and nothing is launched.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array and it keeps the last call's contents.  The per-unit
 * arrival counts are the only part that must start at zero: each call clears
 * them on its stream (one cudaMemsetAsync of B * H_kv * 8 bytes) before its
 * kernel, so a call that follows a timed-out one, or a call of another
 * context whose partials overlapped these counts, starts clean.  Calls whose
 * kernels overlap on the GPU (e.g. on unordered streams) race on the array.
 * The address looked up is that of the device's current context; it is not
 * looked up again after a device reset. */
fkv_status fkv_decode_attn_noalloc(fkv_ctx* ctx, const void* q, int layer, int mode,
                                   const int32_t* seq_lens, void* out, void* stream);

/* Causal prefill attention of a layer over a prompt occupying cache rows
 * [0, S) of every sequence (the storage caches already hold those rows).
 * This is the attention kernel whose throughput and time to first token the
 * FusedKV slides compare across methods ("Prefill improves while kernel
 * throughput falls", Fig.4; reading notes §2.5); the upper layers' K/V follow
 * Eqs.(4)-(6) as in fkv_decode_attn.
 * q: device [B, H_q, S, D]; out: device [B, H_q, S, D]; context dtype.
 * Query row m sees key rows t <= m.  Modes and sources as for decode; fused
 * K/V tiles are built while staging them for the tensor cores.
 * Requires dtype FKV_BF16 (FKV_ERR_UNSUPPORTED otherwise); 1 <= S <= S_max. */
fkv_status fkv_prefill_attn(fkv_ctx* ctx, const void* q, int layer, int mode, int S,
                            void* out, void* stream);

/* Causal prefill of a chunk of C prompt positions q_start .. q_start+C-1 over
 * an existing cache (a long prompt processed in chunks, or a prompt that
 * extends a cached prefix).  The rows [0, q_start + C) of the caches the call
 * reads must already hold the prompt's keys and values (fkv_append_kv); query
 * row i of the chunk sees cache rows t <= q_start + i.
 * q: device [B, H_q, C, D]; out: device [B, H_q, C, D]; bf16.
 * fkv_prefill_attn(S) is this call with q_start = 0 and C = S.  The first
 * token after a prompt of S positions -- the only upper-layer position time to
 * first token needs (FusedKV slides, backup "prefill skipping has a specific
 * scope"; reading notes §2.5) -- is one fkv_decode_attn call with length S.
 * Errors: FKV_ERR_INVALID_ARG unless C >= 1, q_start >= 0 and
 * q_start + C <= S_max; otherwise as fkv_prefill_attn. */
fkv_status fkv_prefill_attn_chunk(fkv_ctx* ctx, const void* q, int layer, int mode, int q_start,
                                  int C, void* out, void* stream);

/* Synchronise the stream, then report and clear the device status word:
 * FKV_OK, FKV_ERR_DEVICE_ARG or FKV_ERR_TIMEOUT (FKV_ERR_CUDA if the sync
 * itself fails). */
fkv_status fkv_get_device_status(fkv_ctx* ctx, void* stream);

/* For tests of the failure path only (the paper has no counterpart).  Sets
 * the wall-clock limit, in ns, of every bounded device wait of this context's
 * later kernels (fkv_create sets 1 s, the maximum accepted).  0 makes every
 * wait report a timeout at once, which takes each kernel down its timeout
 * path at its first wait, on a kernel that does no out-of-bounds access: it records
 * FKV_ERR_TIMEOUT, lets its copies and products in flight finish (with their
 * own fixed limit), frees its tensor memory and returns, leaving some outputs
 * unwritten.  The limit lives in device memory, so replays of captured graphs
 * read the current value.  Synchronous (cudaMemcpy): not during a stream
 * capture.  FKV_ERR_INVALID_ARG above 1 s. */
fkv_status fkv_set_wait_limit(fkv_ctx* ctx, unsigned long long limit_ns);

/* A static, human-readable name of a status code. */
const char* fkv_status_string(fkv_status s);

#ifdef __cplusplus
}
#endif

#endif /* FUSEDKV_H_ */
