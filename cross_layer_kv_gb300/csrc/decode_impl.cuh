// Split-K flash-decoding for FusedKV upper-layer attention (and the vanilla /
// Lite paths), sm_103a.
//
// What one call computes (FusedKV slides, Eqs.(4)-(6); reading notes §2.3):
// for every sequence b and query head h (KV head kh = h / G)
//     s_t = scale * q_h . K_t,  t < len[b]
//     o_h = sum_t softmax(s)_t V_t
// with K_t / V_t the layer's own rows (vanilla), K^n / V^1 (lite), or
// a_1 (.) K^1_t + a_n (.) K^n_t and b_1 (.) V^1_t + b_n (.) V^n_t (fused).
//
// Design (GB300):
//  * Every warp is an independent streaming worker.  The (b, kh, t) rows of
//    the whole call, sum_b H_kv * len[b], are cut into equal contiguous ranges,
//    one per warp of the grid (balanced for ragged lengths).  A warp's range
//    crosses at most a few (b, kh) units; for each unit it touches it writes
//    one partial (m, l, o) per query head of the group.
//  * A warp streams its rows tile by tile with cp.async.bulk (TMA bulk copies)
//    into a private ring of NS shared-memory stages, completion tracked by one
//    mbarrier per stage; lane 0 refills a stage as soon as the warp has read
//    it.  No CTA-wide barrier in the main loop.
//  * Lane mapping: a row of D elements is C = D*sizeof(T)/16 chunks of 16
//    bytes; lane = g*C + c handles chunk c of row g of each R = 32/C row step,
//    so a warp reads contiguous shared memory (conflict-free) for every D.
//  * Fusion stays in registers and costs no extra arithmetic per byte:
//      q . (a_1 (.) K^1 + a_n (.) K^n) = (q (.) a_1) . K^1 + (q (.) a_n) . K^n
//      sum_t p_t (b_1 (.) V^1_t + b_n (.) V^n_t)
//          = b_1 (.) sum_t p_t V^1_t + b_n (.) sum_t p_t V^n_t
//    q is pre-scaled once per unit; two fp32 accumulators take the two value
//    sources and b is applied once when the partial is written.  Nothing
//    reconstructed is written to memory.
//  * All G query heads of a KV head share each tile read (GQA reuse); online
//    softmax in base 2 with warp-shuffle reductions.
//  * The warp that writes the last partial of a (b, kh) unit merges the
//    unit's partials with their log-sum-exp weights and writes the output
//    rows, so one call is one kernel.  Arrivals are counted per unit in a
//    64-bit word tagged with the call's epoch: a count left by an earlier call
//    (or by a call that stopped early) carries another epoch and restarts, so
//    the workspace never needs clearing.  The merging warp clears its unit's
//    word, so a launch replayed from a CUDA graph (same epoch) starts afresh.
#pragma once

#include <cfloat>
#include <cstdint>

#include "fkv_device.cuh"
#include "fkv_kernels.h"

namespace fkv {

// Launch shape of the decode kernel per element type, head dim, source count
// and group size: W warps per CTA, NS ring stages per warp, SB bytes per stage,
// VEC 16-byte chunks per lane.  Chosen from launch-shape sweeps on GB300 at the
// 332M (D=64), 4B (D=80) and 1.5B (D=128) workloads:
//  * power-of-two rows (128 / 256 bytes): 8 warps; one source streams best
//    from 2 x 12 KB stages, two sources from 3 x 8 KB;
//  * 160 / 192-byte rows (D = 80, 96): 2 chunks per lane (5 or 6 lanes per
//    row instead of 10 or 12, so 2.5x fewer shuffles per row); one source
//    with 16 warps x 2 x 6 KB, two sources with 8 warps x 2 x 12 KB (their
//    registers do not fit the 128 a thread gets at 16 warps);
//  * G = 4 or fp32 rows wider than 256 bytes: 8 warps x 3 x 8 KB, 1 chunk.
// Every shape keeps 96-192 KB of loads in flight per SM.
// FKV_DECODE_{WARPS,STAGES,STAGE_BYTES,VEC} override all shapes at build time
// (for tuning sweeps).
template <typename T, int D, int NSRC, int G>
struct DecodeShape {
  static constexpr int ROWB = D * (int)sizeof(T);
  static constexpr bool pow2 = ROWB == 128 || ROWB == 256;
  static constexpr bool odd = (ROWB == 160 || ROWB == 192) && G <= 2;
  static constexpr int W0 = odd && NSRC == 1 ? 16 : 8;
  static constexpr int NS0 = (pow2 && NSRC == 2) || (!pow2 && !odd) ? 3 : 2;
  static constexpr int SB0 = NS0 == 3 ? 8192 : (W0 == 16 ? 6144 : 12288);
  static constexpr int VEC0 = odd ? 2 : 1;
#ifdef FKV_DECODE_WARPS
  static constexpr int W = FKV_DECODE_WARPS;
#else
  static constexpr int W = W0;
#endif
#ifdef FKV_DECODE_STAGES
  static constexpr int NS = FKV_DECODE_STAGES;
#else
  static constexpr int NS = NS0;
#endif
#ifdef FKV_DECODE_STAGE_BYTES
  static constexpr int SB = FKV_DECODE_STAGE_BYTES;
#else
  static constexpr int SB = SB0;
#endif
#ifdef FKV_DECODE_VEC
  static constexpr int VEC = ROWB % (16 * FKV_DECODE_VEC) == 0 ? FKV_DECODE_VEC : 1;
#else
  static constexpr int VEC = VEC0;
#endif
};

template <typename T, int D, int NSRC, int SB, int VEC>
struct DecodeCfg {
  static constexpr int ROWB = D * (int)sizeof(T);   // bytes per cache row
  static constexpr int C = ROWB / (16 * VEC);        // lanes per row (VEC 16-byte chunks each)
  static constexpr int R = 32 / C;                   // rows per warp step
  static constexpr int EC = 16 / (int)sizeof(T);     // elements per 16-byte chunk
  static constexpr int E = EC * VEC;                 // elements per lane
  static constexpr int STAGE_TARGET = SB;             // bytes per stage (all tensors)
  static constexpr int STEPS_RAW = STAGE_TARGET / (2 * NSRC * R * ROWB);
  static constexpr int STEPS = STEPS_RAW < 1 ? 1 : STEPS_RAW;
  static constexpr int TR = R * STEPS;               // rows per tile
  static constexpr int TILE_BYTES = TR * ROWB;       // one tensor's tile
  static constexpr int STAGE_BYTES = 2 * NSRC * TILE_BYTES;
  static_assert(ROWB % (16 * VEC) == 0, "row must split into whole lane chunks");
  static_assert(C >= 1 && C <= 32, "row must fit one warp of 16-byte chunks");
};

// Partial record of one (slot, query head): o[D] then m, l (padded to 4).
__host__ __device__ constexpr int partial_stride(int D) { return D + 4; }

struct SplitParams {
  const void* k0;
  const void* k1;
  const void* v0;
  const void* v1;
  const float* a0;
  const float* a1;
  const float* b0;
  const float* b1;
  const void* q;
  void* out;
  const int32_t* seq_lens;
  float* ws;                       // partials
  unsigned long long* counters;    // one arrival word per (b, kh) unit
  int* status;
  const unsigned long long* wait_limit;  // limit of the bounded waits (device word)
  int B, H_kv, S_max;
  int window;                      // > 0: only the last `window` rows of each sequence
  int ring;                        // > 0: caches are rings of this many rows (position % ring)
  unsigned epoch;                  // tag of this call's arrivals
  float qscale;  // softmax scale * log2(e)
};

// Walk of a warp's row range, one tile at a time, crossing (b, kh) units.
struct RowWalker {
  long long r, r1;
  int b, h, t;

  __device__ __forceinline__ bool next(const int* lens, int H_kv, int B, int TR, int& tb, int& th,
                                       int& tt, int& tn, bool& last) {
    if (r >= r1) return false;
    const int L = lens[b];
    const long long seg = min((long long)(L - t), r1 - r);
    const int n = (int)min((long long)TR, seg);
    tb = b;
    th = h;
    tt = t;
    tn = n;
    last = (n == seg);
    t += n;
    r += n;
    if (t == L) {
      t = 0;
      if (++h == H_kv) {
        h = 0;
        ++b;
        while (r < r1 && b < B && lens[b] == 0) ++b;
      }
    }
    return true;
  }
};

// VEC consecutive 16-byte chunks of shared memory -> fp32.
template <typename T, int VEC>
__device__ __forceinline__ void load_chunks(const uint8_t* src, float* f) {
#pragma unroll
  for (int v = 0; v < VEC; ++v)
    unpack16<T>(*reinterpret_cast<const uint4*>(src + 16 * v), f + v * (16 / (int)sizeof(T)));
}

// (c0, c1) += (a0, a1) * (b0, b1) with one packed fp32 FMA (fma.rn.f32x2).
__device__ __forceinline__ void fma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\t"
      "mov.b64 B, {%4, %5};\n\t"
      "mov.b64 C, {%0, %1};\n\t"
      "fma.rn.f32x2 C, A, B, C;\n\t"
      "mov.b64 {%0, %1}, C;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Sum over the C lanes of each row group; every lane of the group gets it.
template <int C>
__device__ __forceinline__ float group_sum(float v, int lane) {
  if constexpr ((C & (C - 1)) == 0) {
#pragma unroll
    for (int o = C / 2; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  } else {
    const int c = lane % C;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float u = __shfl_down_sync(0xffffffffu, v, o);
      if (o < C && c + o < C) v += u;
    }
    return __shfl_sync(0xffffffffu, v, lane - c);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Count one arrival on a unit's word for call `epoch`; returns the count of
// this epoch including this arrival (0 if the retry bound ran out).  A word
// holding another epoch restarts at 1.
__device__ __forceinline__ unsigned unit_arrive(unsigned long long* word, unsigned epoch) {
  unsigned long long old = atomicAdd(word, 0ull);
#pragma unroll 1
  for (int i = 0; i < (1 << 20); ++i) {
    const unsigned long long nv = (unsigned)(old >> 32) == epoch
                                      ? old + 1ull
                                      : (((unsigned long long)epoch << 32) | 1ull);
    const unsigned long long prev = atomicCAS(word, old, nv);
    if (prev == old) return (unsigned)(nv & 0xffffffffull);
    old = prev;
  }
  return 0;
}

// Merge the partials of unit (b, h) -- written by warps wf..wl at slots
// w + u, skipping the warps with empty ranges -- into the G output rows.  One
// warp; partials are read through L2 (__ldcg), since other SMs wrote them in
// this launch.  Lane i takes the (m, l) of partial i of a batch of 32, and
// the o rows of MB partials (8, or fewer where registers are tight) are
// loaded at once for all G heads, so a merge
// of up to 32 partials costs two dependent L2 round trips rather than one per
// partial and head.
template <typename T, int D, int G, int MB = (G * ((D + 31) / 32) <= 4 ? 8 : 4)>
__device__ __forceinline__ void merge_unit(const float* ws, T* out, long long u, long long wf,
                                           long long wl, long long N, long long total, int b,
                                           int h, int H, int lane) {
  constexpr int PS = partial_stride(D);
  constexpr int DPL = (D + 31) / 32;
  const float* base = ws + (size_t)(wf + u) * G * PS;
  const int P = (int)(wl - wf + 1);
  float M[G], L[G], acc[G][DPL];
  float m0[G], l0[G];  // (m, l) of this lane's partial in the first batch
#pragma unroll
  for (int hq = 0; hq < G; ++hq) {
    M[hq] = -FLT_MAX;
    m0[hq] = -FLT_MAX;
    l0[hq] = 0.f;
  }
  for (int p0 = 0; p0 < P; p0 += 32) {
    const long long w = wf + p0 + lane;
    if (p0 + lane < P && w * total / N < (w + 1) * total / N) {
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        const float* rec = base + ((size_t)(p0 + lane) * G + hq) * PS;
        const float mv = __ldcg(rec + D);
        if (p0 == 0) {
          m0[hq] = mv;
          l0[hq] = __ldcg(rec + D + 1);
        }
        M[hq] = fmaxf(M[hq], mv);
      }
    }
  }
#pragma unroll
  for (int hq = 0; hq < G; ++hq) {
    M[hq] = warp_max(M[hq]);
    L[hq] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[hq][k] = 0.f;
  }
  for (int p0 = 0; p0 < P; p0 += 32) {
    const long long w = wf + p0 + lane;
    const bool ok = p0 + lane < P && w * total / N < (w + 1) * total / N;
    float sc[G];
#pragma unroll
    for (int hq = 0; hq < G; ++hq) {
      sc[hq] = 0.f;
      if (ok) {
        const float* rec = base + ((size_t)(p0 + lane) * G + hq) * PS;
        const float mv = p0 == 0 ? m0[hq] : __ldcg(rec + D);
        const float lv = p0 == 0 ? l0[hq] : __ldcg(rec + D + 1);
        sc[hq] = exp2f(mv - M[hq]);
        L[hq] += sc[hq] * lv;
      }
    }
    const int cnt = min(32, P - p0);
#pragma unroll 1
    for (int i0 = 0; i0 < cnt; i0 += MB) {
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const int i = i0 + j;
#pragma unroll
        for (int hq = 0; hq < G; ++hq) {
          const float si = __shfl_sync(0xffffffffu, sc[hq], i & 31);
          const bool take = i < cnt && si != 0.f;
          const float* rec = base + ((size_t)(p0 + i) * G + hq) * PS;
#pragma unroll
          for (int k = 0; k < DPL; ++k) {
            const int d = lane + 32 * k;
            float x = 0.f;
            if (take && d < D) x = __ldcg(rec + d);
            acc[hq][k] = fmaf(si, x, acc[hq][k]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int hq = 0; hq < G; ++hq) {
    const float inv = 1.f / warp_sum(L[hq]);
    T* orow = out + ((size_t)b * H * G + (size_t)h * G + hq) * D;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const int d = lane + 32 * k;
      if (d < D) {
        if constexpr (sizeof(T) == 4) orow[d] = acc[hq][k] * inv;
        else orow[d] = __float2bfloat16_rn(acc[hq][k] * inv);
      }
    }
  }
}

// Shared-memory bytes of the split kernel besides the stages.
__host__ __device__ constexpr size_t decode_aux_bytes(int warps, int stages, int B) {
  return (size_t)warps * stages * 8 + (size_t)(3 * B + 2) * 4;
}

// WGT: a single source scaled by channel weights (q (.) a before the dot
// products, b on the value sums); always set for two sources.
template <typename T, int D, int NSRC, bool WGT, int G, int W, int NS, int SB, int VEC>
__global__ void __launch_bounds__(W * 32, 1) decode_split_kernel(const SplitParams p) {
  using Cfg = DecodeCfg<T, D, NSRC, SB, VEC>;
  constexpr int C = Cfg::C, R = Cfg::R, E = Cfg::E, TR = Cfg::TR, STEPS = Cfg::STEPS;
  constexpr int EC = Cfg::EC;
  constexpr int ROWB = Cfg::ROWB, TILE = Cfg::TILE_BYTES, STAGE = Cfg::STAGE_BYTES;
  constexpr int PS = partial_stride(D);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)W * NS * STAGE);
  int* lens = reinterpret_cast<int*>(bars + W * NS);  // rows attended per sequence
  int* pre = lens + p.B;      // pre[b] = sum_{b' < b} lens[b'], B + 1 entries
  int* first = pre + p.B + 1; // cache row of each sequence's first attended row

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bars[warp * NS + s], 1);
    fence_mbar_init();
  }
  grid_dep_trigger();
  grid_dep_wait();
  const unsigned long long wlim = wait_limit_ns(p.wait_limit);

  // Sequence lengths, clamped to [0, S_max]; one CTA reports bad ones.
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
    int L = p.seq_lens[i];
    if (L < 1 || L > p.S_max) {
      if (blockIdx.x == 0) flag_status(p.status, kDevBadArg);
      L = L < 0 ? 0 : (L > p.S_max ? p.S_max : L);
    }
    // a sliding-window layer attends to the last `window` rows only
    const int Le = p.window > 0 && L > p.window ? p.window : L;
    lens[i] = Le;
    // cache row of the first attended position (in a ring: its row, so that
    // the copies below need no division)
    first[i] = p.ring > 0 ? (L - Le) % p.ring : L - Le;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int x = base + lane < p.B ? lens[base + lane] : 0;
      int incl = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (base + lane < p.B) pre[base + lane] = run + incl - x;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre[p.B] = run;
  }
  __syncthreads();

  const int H = p.H_kv;
  if (blockIdx.x == 0) {
    // sequences of length 0 have no rows and so no merging warp: zero output
    const int row_elems = H * G * D;
    for (int bb = 0; bb < p.B; ++bb) {
      if (lens[bb] != 0) continue;
      for (int i = threadIdx.x; i < row_elems; i += blockDim.x) {
        const size_t o = (size_t)bb * row_elems + i;
        if constexpr (sizeof(T) == 4) static_cast<float*>(p.out)[o] = 0.f;
        else static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
      }
    }
  }
  const long long total = (long long)H * pre[p.B];
  const long long N = (long long)gridDim.x * W;
  const long long w = (long long)blockIdx.x * W + warp;
  const long long r0 = w * total / N, r1 = (w + 1) * total / N;
  if (r0 >= r1) return;

  // Locate the unit holding row r0: the first b with H * pre[b + 1] > r0.
  RowWalker walk;
  {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((long long)H * pre[mid + 1] > r0) hi = mid; else lo = mid + 1;
    }
    const long long off = r0 - (long long)H * pre[lo];
    const int L = lens[lo];
    walk.b = lo;
    walk.h = (int)(off / L);
    walk.t = (int)(off - (long long)walk.h * L);
    walk.r = r0;
    walk.r1 = r1;
  }
  RowWalker prod = walk;

  uint8_t* wring = smem + (size_t)warp * NS * STAGE;   // this warp's stages
  uint64_t* wbars = bars + warp * NS;
  const uint64_t policy = l2_policy_evict_first();
  const size_t row_stride_u = (size_t)(p.ring > 0 ? p.ring : p.S_max) * ROWB;  // bytes per unit

  auto issue = [&](int stage, int b, int h, int t, int n) {
    if (lane == 0) {
      uint8_t* dst = wring + (size_t)stage * STAGE;
      uint64_t* bar = &wbars[stage];
      const size_t base = ((size_t)b * H + h) * row_stride_u;
      const uint32_t bytes = (uint32_t)n * ROWB;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, bytes * 2 * NSRC);
      if (p.ring == 0) {
        // rows first + t .. + n - 1 of the unit's plane
        const size_t off = base + (size_t)(first[b] + t) * ROWB;
        bulk_g2s(dst, static_cast<const uint8_t*>(p.k0) + off, bytes, bar, policy);
        if constexpr (NSRC == 2)
          bulk_g2s(dst + TILE, static_cast<const uint8_t*>(p.k1) + off, bytes, bar, policy);
        bulk_g2s(dst + NSRC * TILE, static_cast<const uint8_t*>(p.v0) + off, bytes, bar, policy);
        if constexpr (NSRC == 2)
          bulk_g2s(dst + 3 * TILE, static_cast<const uint8_t*>(p.v1) + off, bytes, bar, policy);
      } else {
        // a ring cache: the rows may wrap past its end (t < window <= ring,
        // so at most once), and then take a second copy from its start
        int r0 = first[b] + t;
        if (r0 >= p.ring) r0 -= p.ring;
        const int n1 = r0 + n > p.ring ? p.ring - r0 : n;
        const size_t off = base + (size_t)r0 * ROWB;
        const uint32_t b1 = (uint32_t)n1 * ROWB, b2 = bytes - b1;
        const void* src[2 * NSRC];
        src[0] = p.k0;
        src[NSRC] = p.v0;
        if constexpr (NSRC == 2) {
          src[1] = p.k1;
          src[3] = p.v1;
        }
#pragma unroll
        for (int i = 0; i < 2 * NSRC; ++i) {
          bulk_g2s(dst + i * TILE, static_cast<const uint8_t*>(src[i]) + off, b1, bar, policy);
          if (b2)
            bulk_g2s(dst + i * TILE + b1, static_cast<const uint8_t*>(src[i]) + base, b2, bar, policy);
        }
      }
    }
  };

  int issued = 0;
#pragma unroll 1
  for (int s = 0; s < NS; ++s) {
    int tb, th, tt, tn;
    bool tl;
    if (!prod.next(lens, H, p.B, TR, tb, th, tt, tn, tl)) break;
    issue(s, tb, th, tt, tn);
    ++issued;
  }

  const int g = lane / C, c = lane % C;
  const bool active = g < R;

  float qa[G][E];                       // q (.) a_first * scale * log2 e
  float qb[NSRC == 2 ? G : 1][E];       // q (.) a_second * scale * log2 e
  float o0[G][E];
  float o1[NSRC == 2 ? G : 1][E];
  float m[G], l[G];
  bool fresh = true;
  int consumed = 0;

#pragma unroll 1
  for (;;) {
    int b, h, t0, n;
    bool last;
    if (!walk.next(lens, H, p.B, TR, b, h, t0, n, last)) break;
    const int stage = consumed % NS;
    const uint32_t parity = (uint32_t)(consumed / NS) & 1u;

    if (fresh) {
      // Query (and key weights) of this (b, kh) unit, chunk c of every head.
      const T* qp = static_cast<const T*>(p.q) + ((size_t)b * H * G + (size_t)h * G) * D + c * E;
      float wa0[E], wa1[E];
#pragma unroll
      for (int e = 0; e < E; ++e) { wa0[e] = 1.f; wa1[e] = 1.f; }
      if constexpr (NSRC == 2) {
        const float* ap = p.a0 + (size_t)h * D + c * E;
        const float* an = p.a1 + (size_t)h * D + c * E;
#pragma unroll
        for (int e = 0; e < E; ++e) { wa0[e] = ap[e]; wa1[e] = an[e]; }
      } else if (WGT) {  // single source with channel scaling
        const float* ap = p.a0 + (size_t)h * D + c * E;
#pragma unroll
        for (int e = 0; e < E; ++e) wa0[e] = ap[e];
      }
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        float qf[E];
#pragma unroll
        for (int v = 0; v < VEC; ++v)
          unpack16<T>(*reinterpret_cast<const uint4*>(qp + (size_t)hq * D + v * EC), qf + v * EC);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          qa[hq][e] = qf[e] * p.qscale * wa0[e];
          if constexpr (NSRC == 2) qb[hq][e] = qf[e] * p.qscale * wa1[e];
          o0[hq][e] = 0.f;
          if constexpr (NSRC == 2) o1[hq][e] = 0.f;
        }
        m[hq] = -FLT_MAX;
        l[hq] = 0.f;
      }
      fresh = false;
    }

    // warp-uniform: every lane leaves, or none does (shuffles follow)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&wbars[stage], parity, wlim))) {
      flag_status(p.status, kDevTimeout);
      // Let the copies still in flight land before the CTA can exit: every
      // stage issued and not yet consumed, the one just awaited included.
      for (int k = consumed; k < issued; ++k)
        (void)mbar_wait_bounded(&wbars[k % NS], (uint32_t)(k / NS) & 1u, kDrainLimitNs);
      return;
    }

    const uint8_t* st = wring + (size_t)stage * STAGE;
    const uint8_t* kt0 = st;
    const uint8_t* kt1 = st + TILE;
    const uint8_t* vt0 = st + NSRC * TILE;
    const uint8_t* vt1 = st + (NSRC + 1) * TILE;

    // Scores of the tile: step j covers rows j*R .. j*R+R-1.
    float s[STEPS][G];
#pragma unroll
    for (int j = 0; j < STEPS; ++j) {
      const int row = j * R + g;
      float acc[G], acc2[G];
#pragma unroll
      for (int hq = 0; hq < G; ++hq) acc[hq] = acc2[hq] = 0.f;
      if (active) {
        float kf[E];
        load_chunks<T, VEC>(kt0 + row * ROWB + c * 16 * VEC, kf);
#pragma unroll
        for (int hq = 0; hq < G; ++hq)
#pragma unroll
          for (int e = 0; e < E; e += 2)
            fma2(acc[hq], acc2[hq], qa[hq][e], qa[hq][e + 1], kf[e], kf[e + 1]);
        if constexpr (NSRC == 2) {
          load_chunks<T, VEC>(kt1 + row * ROWB + c * 16 * VEC, kf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq)
#pragma unroll
            for (int e = 0; e < E; e += 2)
              fma2(acc[hq], acc2[hq], qb[hq][e], qb[hq][e + 1], kf[e], kf[e + 1]);
        }
#pragma unroll
        for (int hq = 0; hq < G; ++hq) acc[hq] += acc2[hq];
      }
      const bool ok = active && row < n;
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        const float v = group_sum<C>(acc[hq], lane);
        s[j][hq] = ok ? v : -FLT_MAX;
      }
    }

    // Online softmax: new running max per head (warp-uniform).
#pragma unroll
    for (int hq = 0; hq < G; ++hq) {
      float mt = s[0][hq];
#pragma unroll
      for (int j = 1; j < STEPS; ++j) mt = fmaxf(mt, s[j][hq]);
      mt = warp_max(mt);
      if (mt > m[hq]) {
        const float alpha = fast_exp2(m[hq] - mt);
        l[hq] *= alpha;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          o0[hq][e] *= alpha;
          if constexpr (NSRC == 2) o1[hq][e] *= alpha;
        }
        m[hq] = mt;
      }
    }

    // Values.
#pragma unroll
    for (int j = 0; j < STEPS; ++j) {
      const int row = j * R + g;
      if (active && row < n) {
        float pj[G];
#pragma unroll
        for (int hq = 0; hq < G; ++hq) {
          pj[hq] = fast_exp2(s[j][hq] - m[hq]);
          l[hq] += pj[hq];
        }
        float vf[E];
        load_chunks<T, VEC>(vt0 + row * ROWB + c * 16 * VEC, vf);
#pragma unroll
        for (int hq = 0; hq < G; ++hq)
#pragma unroll
          for (int e = 0; e < E; e += 2)
            fma2(o0[hq][e], o0[hq][e + 1], pj[hq], pj[hq], vf[e], vf[e + 1]);
        if constexpr (NSRC == 2) {
          load_chunks<T, VEC>(vt1 + row * ROWB + c * 16 * VEC, vf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq)
#pragma unroll
            for (int e = 0; e < E; e += 2)
              fma2(o1[hq][e], o1[hq][e + 1], pj[hq], pj[hq], vf[e], vf[e + 1]);
        }
      }
    }

    ++consumed;
    __syncwarp();
    // Refill the stage just read with the warp's next tile.
    {
      int tb, th, tt, tn;
      bool tl;
      if (prod.next(lens, H, p.B, TR, tb, th, tt, tn, tl)) {
        issue(stage, tb, th, tt, tn);
        ++issued;
      }
    }

    if (last) {
      // Combine the R row groups, apply the value weights, write the partial.
      const long long u = (long long)b * H + h;
      float* rec = p.ws + ((size_t)(w + u) * G) * PS;
      float wb0[E], wb1[E];
      constexpr bool scale_v = NSRC == 2 || WGT;
      if constexpr (NSRC == 2) {
        const float* bp = p.b0 + (size_t)h * D + c * E;
        const float* bn = p.b1 + (size_t)h * D + c * E;
#pragma unroll
        for (int e = 0; e < E; ++e) { wb0[e] = bp[e]; wb1[e] = bn[e]; }
      } else if constexpr (scale_v) {
        const float* bp = p.b0 + (size_t)h * D + c * E;
#pragma unroll
        for (int e = 0; e < E; ++e) wb0[e] = bp[e];
      }
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        float lt = 0.f;
#pragma unroll
        for (int k = 0; k < R; ++k) lt += __shfl_sync(0xffffffffu, l[hq], k * C);
        float ov[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          float x0 = 0.f, x1 = 0.f;
#pragma unroll
          for (int k = 0; k < R; ++k) {
            x0 += __shfl_sync(0xffffffffu, o0[hq][e], k * C + c);
            if constexpr (NSRC == 2) x1 += __shfl_sync(0xffffffffu, o1[hq][e], k * C + c);
          }
          if constexpr (NSRC == 2) ov[e] = wb0[e] * x0 + wb1[e] * x1;
          else if constexpr (scale_v) ov[e] = wb0[e] * x0;
          else ov[e] = x0;
        }
        if (g == 0) {
          float4* dst = reinterpret_cast<float4*>(rec + (size_t)hq * PS + c * E);
#pragma unroll
          for (int e = 0; e < E; e += 4) dst[e / 4] = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
        }
        if (lane == 0) {
          rec[(size_t)hq * PS + D] = m[hq];
          rec[(size_t)hq * PS + D + 1] = lt;
        }
      }
      fresh = true;

      // Publish the partial, count the arrival; the last warp of the unit merges.
      const long long su = (long long)H * pre[b] + (long long)h * lens[b];
      const long long eu = su + lens[b];
      const long long wf = ((su + 1) * N - 1) / total, wl = (eu * N - 1) / total;
      int need = 0;
      for (long long w0 = wf; w0 <= wl; w0 += 32) {
        const long long ww = w0 + lane;
        need += __popc(__ballot_sync(0xffffffffu,
                                     ww <= wl && ww * total / N < (ww + 1) * total / N));
      }
      __threadfence();
      __syncwarp();
      unsigned arrived = 0;
      if (lane == 0) arrived = unit_arrive(p.counters + u, p.epoch);
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived == 0) flag_status(p.status, lane == 0 ? kDevTimeout : 0);
      if (arrived == (unsigned)need) {
        // No arrival of this call can follow: clear the word, so that a call
        // with the same epoch (a CUDA graph replaying this launch) starts at 1.
        if (lane == 0) p.counters[u] = 0ull;
        __threadfence();
        // (16-warp shapes have 128 registers a thread: two partials at a time)
        merge_unit<T, D, G, (W > 8 ? 2 : (G * ((D + 31) / 32) <= 4 ? 8 : 4))>(
            p.ws, static_cast<T*>(p.out), u, wf, wl, N, total, b, h, H, lane);
      }
    }
  }
}

template <typename T, int D, int NSRC, int G>
size_t decode_smem_bytes(int B) {
  using S = DecodeShape<T, D, NSRC, G>;
  using Cfg = DecodeCfg<T, D, NSRC, S::SB, S::VEC>;
  return (size_t)S::W * S::NS * Cfg::STAGE_BYTES + decode_aux_bytes(S::W, S::NS, B);
}

template <typename T, int D, int NSRC, bool WGT, int G>
cudaError_t decode_launch_t(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  SplitParams sp;
  sp.k0 = a.k[0];
  sp.k1 = a.k[1];
  sp.v0 = a.v[0];
  sp.v1 = a.v[1];
  sp.a0 = a.a[0];
  sp.a1 = a.a[1];
  sp.b0 = a.b[0];
  sp.b1 = a.b[1];
  sp.q = a.q;
  sp.out = a.out;
  sp.seq_lens = a.seq_lens;
  sp.ws = a.workspace;
  sp.counters = reinterpret_cast<unsigned long long*>(
      reinterpret_cast<char*>(a.workspace) + plan.partial_bytes);
  sp.status = a.status;
  sp.wait_limit = a.wait_limit;
  sp.epoch = a.epoch;
  sp.B = a.batch;
  sp.H_kv = a.kv_heads;
  sp.S_max = a.max_seq;
  sp.window = a.window;
  sp.ring = a.ring;
  sp.qscale = a.softmax_scale * 1.4426950408889634f;
  using S = DecodeShape<T, D, NSRC, G>;
  auto kern = decode_split_kernel<T, D, NSRC, WGT || NSRC == 2, G, S::W, S::NS, S::SB, S::VEC>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem_bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(plan.ctas), dim3(S::W * 32), plan.smem_bytes, stream, sp);
}

}  // namespace fkv
