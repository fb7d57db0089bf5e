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
//    softmax in base 2 with warp-shuffle reductions; a second kernel merges
//    the partials of each (b, h) with their log-sum-exp weights.
#pragma once

#include <cfloat>
#include <cstdint>

#include "fkv_device.cuh"
#include "fkv_kernels.h"

namespace fkv {

template <typename T, int D, int NSRC>
struct DecodeCfg {
  static constexpr int ROWB = D * (int)sizeof(T);   // bytes per cache row
  static constexpr int C = ROWB / 16;                // 16-byte chunks per row
  static constexpr int R = 32 / C;                   // rows per warp step
  static constexpr int E = 16 / (int)sizeof(T);      // elements per chunk
  static constexpr int STAGE_TARGET = 8192;          // bytes per stage (all tensors)
  static constexpr int STEPS_RAW = STAGE_TARGET / (2 * NSRC * R * ROWB);
  static constexpr int STEPS = STEPS_RAW < 1 ? 1 : STEPS_RAW;
  static constexpr int TR = R * STEPS;               // rows per tile
  static constexpr int TILE_BYTES = TR * ROWB;       // one tensor's tile
  static constexpr int STAGE_BYTES = 2 * NSRC * TILE_BYTES;
  static_assert(ROWB % 16 == 0, "row must be a multiple of 16 bytes");
  static_assert(C >= 1 && C <= 32, "row must fit one warp of 16-byte chunks");
};

constexpr int kDecodeWarps = 8;    // warps per CTA
constexpr int kDecodeStages = 3;   // pipeline stages per warp

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
  const int32_t* seq_lens;
  float* ws;
  int* status;
  int B, H_kv, S_max;
  float qscale;  // softmax scale * log2(e)
};

struct MergeParams {
  const int32_t* seq_lens;
  const float* ws;
  void* out;
  int B, H_kv, G, S_max, D;
  int total_warps;
  int is_f32;
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

// Shared-memory bytes of the split kernel besides the stages.
__host__ __device__ constexpr size_t decode_aux_bytes(int warps, int stages, int B) {
  return (size_t)warps * stages * 8 + (size_t)(2 * B + 2) * 4;
}

template <typename T, int D, int NSRC, int G>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
    decode_split_kernel(const SplitParams p) {
  using Cfg = DecodeCfg<T, D, NSRC>;
  constexpr int C = Cfg::C, R = Cfg::R, E = Cfg::E, TR = Cfg::TR, STEPS = Cfg::STEPS;
  constexpr int ROWB = Cfg::ROWB, TILE = Cfg::TILE_BYTES, STAGE = Cfg::STAGE_BYTES;
  constexpr int NS = kDecodeStages, W = kDecodeWarps;
  constexpr int PS = partial_stride(D);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)W * NS * STAGE);
  int* lens = reinterpret_cast<int*>(bars + W * NS);
  int* pre = lens + p.B;  // pre[b] = sum_{b' < b} lens[b'], B + 1 entries

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bars[warp * NS + s], 1);
    fence_mbar_init();
  }
  grid_dep_trigger();
  grid_dep_wait();

  // Sequence lengths, clamped to [0, S_max]; one CTA reports bad ones.
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
    int L = p.seq_lens[i];
    if (L < 1 || L > p.S_max) {
      if (blockIdx.x == 0) flag_status(p.status, kDevBadArg);
      L = L < 0 ? 0 : (L > p.S_max ? p.S_max : L);
    }
    lens[i] = L;
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

  uint8_t* ring = smem + (size_t)warp * NS * STAGE;
  uint64_t* wbars = bars + warp * NS;
  const uint64_t policy = l2_policy_evict_first();
  const size_t row_stride_u = (size_t)p.S_max * ROWB;  // bytes per (b, kh) unit

  auto issue = [&](int stage, int b, int h, int t, int n) {
    if (lane == 0) {
      const size_t off = ((size_t)b * H + h) * row_stride_u + (size_t)t * ROWB;
      const uint32_t bytes = (uint32_t)n * ROWB;
      uint8_t* dst = ring + (size_t)stage * STAGE;
      uint64_t* bar = &wbars[stage];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, bytes * 2 * NSRC);
      bulk_g2s(dst, static_cast<const uint8_t*>(p.k0) + off, bytes, bar, policy);
      if constexpr (NSRC == 2)
        bulk_g2s(dst + TILE, static_cast<const uint8_t*>(p.k1) + off, bytes, bar, policy);
      bulk_g2s(dst + NSRC * TILE, static_cast<const uint8_t*>(p.v0) + off, bytes, bar, policy);
      if constexpr (NSRC == 2)
        bulk_g2s(dst + 3 * TILE, static_cast<const uint8_t*>(p.v1) + off, bytes, bar, policy);
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
      }
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        float qf[E];
        unpack16<T>(*reinterpret_cast<const uint4*>(qp + (size_t)hq * D), qf);
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

    if (!mbar_wait_bounded(&wbars[stage], parity)) {
      flag_status(p.status, kDevTimeout);
      // Let the copies still in flight land before the CTA can exit.
      for (int k = consumed + 1; k < issued; ++k)
        (void)mbar_wait_bounded(&wbars[k % NS], (uint32_t)(k / NS) & 1u, kDrainLimitNs);
      return;
    }

    const uint8_t* st = ring + (size_t)stage * STAGE;
    const uint8_t* kt0 = st;
    const uint8_t* kt1 = st + TILE;
    const uint8_t* vt0 = st + NSRC * TILE;
    const uint8_t* vt1 = st + (NSRC + 1) * TILE;

    // Scores of the tile: step j covers rows j*R .. j*R+R-1.
    float s[STEPS][G];
#pragma unroll
    for (int j = 0; j < STEPS; ++j) {
      const int row = j * R + g;
      float acc[G];
#pragma unroll
      for (int hq = 0; hq < G; ++hq) acc[hq] = 0.f;
      if (active) {
        float kf[E];
        unpack16<T>(*reinterpret_cast<const uint4*>(kt0 + row * ROWB + c * 16), kf);
#pragma unroll
        for (int hq = 0; hq < G; ++hq)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[hq] = fmaf(qa[hq][e], kf[e], acc[hq]);
        if constexpr (NSRC == 2) {
          unpack16<T>(*reinterpret_cast<const uint4*>(kt1 + row * ROWB + c * 16), kf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[hq] = fmaf(qb[hq][e], kf[e], acc[hq]);
        }
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
        unpack16<T>(*reinterpret_cast<const uint4*>(vt0 + row * ROWB + c * 16), vf);
#pragma unroll
        for (int hq = 0; hq < G; ++hq)
#pragma unroll
          for (int e = 0; e < E; ++e) o0[hq][e] = fmaf(pj[hq], vf[e], o0[hq][e]);
        if constexpr (NSRC == 2) {
          unpack16<T>(*reinterpret_cast<const uint4*>(vt1 + row * ROWB + c * 16), vf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq)
#pragma unroll
            for (int e = 0; e < E; ++e) o1[hq][e] = fmaf(pj[hq], vf[e], o1[hq][e]);
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
      if constexpr (NSRC == 2) {
        const float* bp = p.b0 + (size_t)h * D + c * E;
        const float* bn = p.b1 + (size_t)h * D + c * E;
#pragma unroll
        for (int e = 0; e < E; ++e) { wb0[e] = bp[e]; wb1[e] = bn[e]; }
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
    }
  }
}

// Merge of the partials of each (b, query head): one warp per output row.
template <typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const MergeParams p) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  grid_dep_trigger();
  grid_dep_wait();
  const int Hq = p.H_kv * p.G;
  if (row >= (long long)p.B * Hq) return;
  const int b = (int)(row / Hq), hq = (int)(row % Hq);
  const int h = hq / p.G, hl = hq % p.G;
  const int D = p.D, PS = partial_stride(D);

  auto clamp_len = [&](int L) { return L < 0 ? 0 : (L > p.S_max ? p.S_max : L); };
  long long before = 0, total = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int i = base + lane;
    const long long L = i < p.B ? clamp_len(p.seq_lens[i]) : 0;
    long long x = L, y = i < b ? L : 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      x += __shfl_xor_sync(0xffffffffu, x, o);
      y += __shfl_xor_sync(0xffffffffu, y, o);
    }
    total += x;
    before += y;
  }
  const int Lb = clamp_len(p.seq_lens[b]);
  T* out = static_cast<T*>(p.out) + (size_t)row * D;
  if (Lb == 0) {
    for (int d = lane; d < D; d += 32) {
      if constexpr (sizeof(T) == 4) out[d] = 0.f;
      else out[d] = __float2bfloat16_rn(0.f);
    }
    return;
  }
  const long long H = p.H_kv, N = p.total_warps;
  total *= H;
  const long long su = H * before + (long long)h * Lb, eu = su + Lb;
  const long long u = (long long)b * H + h;
  const long long wf = ((su + 1) * N - 1) / total, wl = (eu * N - 1) / total;

  float M = -FLT_MAX;
  for (long long w = wf; w <= wl; ++w) {
    const long long s0 = w * total / N, s1 = (w + 1) * total / N;
    if (s0 >= s1 || s0 >= eu || s1 <= su) continue;
    M = fmaxf(M, p.ws[((size_t)(w + u) * p.G + hl) * PS + D]);
  }
  float Lsum = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // D <= 128
  for (long long w = wf; w <= wl; ++w) {
    const long long s0 = w * total / N, s1 = (w + 1) * total / N;
    if (s0 >= s1 || s0 >= eu || s1 <= su) continue;
    const float* rec = p.ws + ((size_t)(w + u) * p.G + hl) * PS;
    const float sc = exp2f(rec[D] - M);
    Lsum += sc * rec[D + 1];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int d = lane + 32 * k;
      if (d < D) acc[k] += sc * rec[d];
    }
  }
  const float inv = 1.f / Lsum;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int d = lane + 32 * k;
    if (d < D) {
      if constexpr (sizeof(T) == 4) out[d] = acc[k] * inv;
      else out[d] = __float2bfloat16_rn(acc[k] * inv);
    }
  }
}

template <typename T, int D, int NSRC, int G>
size_t decode_smem_bytes(int B) {
  using Cfg = DecodeCfg<T, D, NSRC>;
  return (size_t)kDecodeWarps * kDecodeStages * Cfg::STAGE_BYTES +
         decode_aux_bytes(kDecodeWarps, kDecodeStages, B);
}

template <typename T, int D, int NSRC, int G>
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
  sp.seq_lens = a.seq_lens;
  sp.ws = a.workspace;
  sp.status = a.status;
  sp.B = a.batch;
  sp.H_kv = a.kv_heads;
  sp.S_max = a.max_seq;
  sp.qscale = a.softmax_scale * 1.4426950408889634f;
  auto kern = decode_split_kernel<T, D, NSRC, G>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(plan.ctas), dim3(kDecodeWarps * 32), plan.smem_bytes, stream, sp);
  if (e != cudaSuccess) return e;

  MergeParams mp;
  mp.seq_lens = a.seq_lens;
  mp.ws = a.workspace;
  mp.out = a.out;
  mp.B = a.batch;
  mp.H_kv = a.kv_heads;
  mp.G = G;
  mp.S_max = a.max_seq;
  mp.D = D;
  mp.total_warps = plan.ctas * kDecodeWarps;
  mp.is_f32 = sizeof(T) == 4;
  const long long rows = (long long)a.batch * a.kv_heads * G;
  return launch_pdl(decode_merge_kernel<T>, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, stream,
                    mp);
}

}  // namespace fkv
