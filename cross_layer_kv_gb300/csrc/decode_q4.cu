// Decode attention over 4-bit caches: dequantisation fused with the
// reconstruction and the softmax, all in registers (FusedKV slides, "Four-bit
// KV quantization is the stronger combination", Table 14: 4-bit KV on top of
// FusedKV; the quantisation grouping is this library's: 16 channels per
// group, bf16 scale and minimum, see append_q4_kernel).
//
// Same structure as decode_split_kernel (per-warp cp.async.bulk rings,
// stream-K row partition, in-kernel log-sum-exp merge); what differs is the
// row format and the arithmetic per lane.  A lane owns one group of 16
// channels of a row (8 bytes of codes, 4 bytes of parameters), so a row takes
// C = D/16 lanes and a warp step covers R = 32/C rows.  The dequantisation is
// folded into the dot products:
//   q . (m + c * s)            = m' * sum(q) + s * (q . (128 + c)),
//   sum_t p_t (m_t + c_t s_t)  = sum_t p_t m'_t + sum_t (p_t s_t) (128 + c_t),
// with m' = m - 128 s per group and row, so each element costs one byte
// permute (128 + c is built exactly in the mantissa) and one packed FMA;
// sum(q) per group is computed once per (b, kv-head) unit.
#include "decode_impl.cuh"

namespace fkv {
namespace {

// Launch shape per source count: warps per CTA, ring stages per warp, bytes
// per stage.  Two sources (fused) need about 255 registers a thread, so 8
// warps; one source fits in 168, so 12 warps fit and hide more latency (at
// 12 x 2 x 9 KB the 332M lite call went 70.5 -> 66.3 us and the 4B one
// 346 -> 302 us against 8 x 2 x 12 KB).  Larger stages spread the per-tile
// work (row-max shuffles, refill, barrier) over more rows.
// FKV_Q4_{WARPS,STAGES,STAGE_BYTES}{1,2} override them at build time (sweeps).
template <int NSRC>
struct Q4Shape;
template <>
struct Q4Shape<1> {
#ifdef FKV_Q4_WARPS1
  static constexpr int W = FKV_Q4_WARPS1, NS = FKV_Q4_STAGES1, SB = FKV_Q4_STAGE_BYTES1;
#else
  static constexpr int W = 12, NS = 2, SB = 9216;
#endif
};
template <>
struct Q4Shape<2> {
#ifdef FKV_Q4_WARPS2
  static constexpr int W = FKV_Q4_WARPS2, NS = FKV_Q4_STAGES2, SB = FKV_Q4_STAGE_BYTES2;
#else
  static constexpr int W = 8, NS = 2, SB = 12288;
#endif
};

template <int D, int NSRC>
struct Q4Cfg {
  static constexpr int ROWB = q4_row_bytes(D);       // bytes per cache row
  static constexpr int C = D / kQ4Group;              // lanes per row
  static constexpr int R = 32 / C;                    // rows per warp step
  static constexpr int E = kQ4Group;                  // channels per lane
  static constexpr int STEPS_RAW = Q4Shape<NSRC>::SB / (2 * NSRC * R * ROWB);
  static constexpr int STEPS = STEPS_RAW < 1 ? 1 : STEPS_RAW;
  static constexpr int TR = R * STEPS;
  static constexpr int TILE_BYTES = TR * ROWB;
  static constexpr int STAGE_BYTES = 2 * NSRC * TILE_BYTES;
};

// 16 four-bit codes (two 32-bit words, channel 2i in the low nibble of byte
// i) -> fp32 values 128 + code, exactly: one byte permute per code places it
// in the mantissa under the exponent of 128 (0x43000000 | code << 16).  The
// bias of 128 is folded into the group minimum by the caller (m - 128 s), so
// no per-element subtraction is needed; products q * (128 + c) keep full
// fp32 accuracy.
__device__ __forceinline__ void codes16_biased(uint32_t w0, uint32_t w1, float* c) {
  const uint32_t ws[2] = {w0, w1};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t lo = ws[k] & 0x0F0F0F0Fu, hi = (ws[k] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      c[8 * k + 2 * b] = __uint_as_float(__byte_perm(lo, 0x43000000u, 0x7054 | (b << 8)));
      c[8 * k + 2 * b + 1] = __uint_as_float(__byte_perm(hi, 0x43000000u, 0x7054 | (b << 8)));
    }
  }
}

__device__ __forceinline__ void q4_params(uint32_t w, float& scale, float& lo) {
  scale = __uint_as_float(w << 16);
  lo = __uint_as_float(w & 0xffff0000u);
}

template <int D, int NSRC, bool WGT, int G>
__global__ void __launch_bounds__(Q4Shape<NSRC>::W * 32, 1) decode_q4_kernel(const SplitParams p) {
  using Cfg = Q4Cfg<D, NSRC>;
  constexpr int C = Cfg::C, R = Cfg::R, E = Cfg::E, TR = Cfg::TR, STEPS = Cfg::STEPS;
  constexpr int ROWB = Cfg::ROWB, TILE = Cfg::TILE_BYTES, STAGE = Cfg::STAGE_BYTES;
  constexpr int NS = Q4Shape<NSRC>::NS, W = Q4Shape<NSRC>::W;
  constexpr int PS = partial_stride(D);

  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)W * NS * STAGE);
  int* lens = reinterpret_cast<int*>(bars + W * NS);
  int* pre = lens + p.B;
  int* first = pre + p.B + 1;

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

  for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
    int L = p.seq_lens[i];
    if (L < 1 || L > p.S_max) {
      if (blockIdx.x == 0) flag_status(p.status, kDevBadArg);
      L = L < 0 ? 0 : (L > p.S_max ? p.S_max : L);
    }
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
    const int row_elems = H * G * D;
    for (int bb = 0; bb < p.B; ++bb) {
      if (lens[bb] != 0) continue;
      for (int i = threadIdx.x; i < row_elems; i += blockDim.x)
        static_cast<__nv_bfloat16*>(p.out)[(size_t)bb * row_elems + i] = __float2bfloat16_rn(0.f);
    }
  }
  const long long total = (long long)H * pre[p.B];
  const long long N = (long long)gridDim.x * W;
  const long long w = (long long)blockIdx.x * W + warp;
  const long long r0 = w * total / N, r1 = (w + 1) * total / N;
  if (r0 >= r1) return;

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

  const int g = lane / C, c = lane % C;   // row in step, channel group
  const bool active = g < R;
  constexpr int NS2 = NSRC == 2 ? 2 : 1;

  float qa[NS2][G][E];     // q (.) a_src * scale * log2 e, per source
  float qsum[NS2][G];      // their sums over the lane's 16 channels
  float oc[NS2][G][E];     // sum_t (p_t s_t) c_t per source
  float om[NS2][G];        // sum_t p_t m_t per source
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
      const __nv_bfloat16* qp =
          static_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * H * G + (size_t)h * G) * D + c * E;
#pragma unroll
      for (int sidx = 0; sidx < NS2; ++sidx) {
        float wa[E];
#pragma unroll
        for (int e = 0; e < E; ++e) wa[e] = 1.f;
        if (NSRC == 2 || WGT) {
          const float* ap = (sidx == 0 ? p.a0 : p.a1) + (size_t)h * D + c * E;
#pragma unroll
          for (int e = 0; e < E; ++e) wa[e] = ap[e];
        }
#pragma unroll
        for (int hq = 0; hq < G; ++hq) {
          float qf[E];
          unpack16<__nv_bfloat16>(*reinterpret_cast<const uint4*>(qp + (size_t)hq * D), qf);
          unpack16<__nv_bfloat16>(*reinterpret_cast<const uint4*>(qp + (size_t)hq * D + 8), qf + 8);
          float sq = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            qa[sidx][hq][e] = qf[e] * p.qscale * wa[e];
            sq += qa[sidx][hq][e];
            oc[sidx][hq][e] = 0.f;
          }
          qsum[sidx][hq] = sq;
          om[sidx][hq] = 0.f;
        }
      }
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        m[hq] = -FLT_MAX;
        l[hq] = 0.f;
      }
      fresh = false;
    }

    // warp-uniform: every lane leaves, or none does (shuffles follow)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&wbars[stage], parity, wlim))) {
      flag_status(p.status, kDevTimeout);
      // let every stage issued and not yet consumed land, this one included
      for (int k = consumed; k < issued; ++k)
        (void)mbar_wait_bounded(&wbars[k % NS], (uint32_t)(k / NS) & 1u, kDrainLimitNs);
      return;
    }

    const uint8_t* st = wring + (size_t)stage * STAGE;

    // scores
    float s[STEPS][G];
#pragma unroll
    for (int j = 0; j < STEPS; ++j) {
      const int row = j * R + g;
      float acc[G];
#pragma unroll
      for (int hq = 0; hq < G; ++hq) acc[hq] = 0.f;
      if (active) {
#pragma unroll
        for (int sidx = 0; sidx < NS2; ++sidx) {
          const uint8_t* rp = st + sidx * TILE + row * ROWB;
          const uint2 cw = *reinterpret_cast<const uint2*>(rp + c * 8);
          float sc, mn;
          q4_params(*reinterpret_cast<const uint32_t*>(rp + D / 2 + c * 4), sc, mn);
          const float mb = fmaf(-128.f, sc, mn);   // x = (m - 128 s) + (128 + c) s
          float cf[E];
          codes16_biased(cw.x, cw.y, cf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq) {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int e = 0; e < E; e += 2)
              fma2(d0, d1, qa[sidx][hq][e], qa[sidx][hq][e + 1], cf[e], cf[e + 1]);
            acc[hq] += mb * qsum[sidx][hq] + sc * (d0 + d1);
          }
        }
      }
      if constexpr ((C & (C - 1)) == 0) {
        const bool ok = active && row < n;
#pragma unroll
        for (int hq = 0; hq < G; ++hq) {
          const float v = group_sum<C>(acc[hq], lane);
          s[j][hq] = ok ? v : -FLT_MAX;
        }
      } else {
#pragma unroll
        for (int hq = 0; hq < G; ++hq) s[j][hq] = acc[hq];
      }
    }
    if constexpr ((C & (C - 1)) != 0) {
      // Rows of 5 or 6 lanes (D = 80, 96) are summed by a five-level shuffle
      // chain and a broadcast: all steps' sums at once, as independent
      // chains whose latencies overlap (at D = 80, 4B-shaped calls: 635 ->
      // 590 us fused, 426 -> 346 us lite; no gain for the two-level sums of
      // 4 or 8 lanes)
#pragma unroll
      for (int j = 0; j < STEPS; ++j) {
        const bool ok = active && j * R + g < n;
#pragma unroll
        for (int hq = 0; hq < G; ++hq) {
          const float v = group_sum<C>(s[j][hq], lane);
          s[j][hq] = ok ? v : -FLT_MAX;
        }
      }
    }

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
        for (int sidx = 0; sidx < NS2; ++sidx) {
          om[sidx][hq] *= alpha;
#pragma unroll
          for (int e = 0; e < E; ++e) oc[sidx][hq][e] *= alpha;
        }
        m[hq] = mt;
      }
    }

    // values
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
#pragma unroll
        for (int sidx = 0; sidx < NS2; ++sidx) {
          const uint8_t* rp = st + (NSRC + sidx) * TILE + row * ROWB;
          const uint2 cw = *reinterpret_cast<const uint2*>(rp + c * 8);
          float sc, mn;
          q4_params(*reinterpret_cast<const uint32_t*>(rp + D / 2 + c * 4), sc, mn);
          const float mb = fmaf(-128.f, sc, mn);
          float cf[E];
          codes16_biased(cw.x, cw.y, cf);
#pragma unroll
          for (int hq = 0; hq < G; ++hq) {
            const float ps = pj[hq] * sc;
            om[sidx][hq] = fmaf(pj[hq], mb, om[sidx][hq]);
#pragma unroll
            for (int e = 0; e < E; e += 2)
              fma2(oc[sidx][hq][e], oc[sidx][hq][e + 1], ps, ps, cf[e], cf[e + 1]);
          }
        }
      }
    }

    ++consumed;
    __syncwarp();
    {
      int tb, th, tt, tn;
      bool tl;
      if (prod.next(lens, H, p.B, TR, tb, th, tt, tn, tl)) {
        issue(stage, tb, th, tt, tn);
        ++issued;
      }
    }

    if (last) {
      const long long u = (long long)b * H + h;
      float* rec = p.ws + ((size_t)(w + u) * G) * PS;
      float wb[NS2][E];
#pragma unroll
      for (int sidx = 0; sidx < NS2; ++sidx) {
#pragma unroll
        for (int e = 0; e < E; ++e) wb[sidx][e] = 1.f;
        if (NSRC == 2 || WGT) {
          const float* bp = (sidx == 0 ? p.b0 : p.b1) + (size_t)h * D + c * E;
#pragma unroll
          for (int e = 0; e < E; ++e) wb[sidx][e] = bp[e];
        }
      }
#pragma unroll
      for (int hq = 0; hq < G; ++hq) {
        float lt = 0.f;
#pragma unroll
        for (int k = 0; k < R; ++k) lt += __shfl_sync(0xffffffffu, l[hq], k * C);
        float ov[E];
#pragma unroll
        for (int e = 0; e < E; ++e) ov[e] = 0.f;
#pragma unroll
        for (int sidx = 0; sidx < NS2; ++sidx) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            float x = 0.f;
#pragma unroll
            for (int k = 0; k < R; ++k)
              x += __shfl_sync(0xffffffffu, oc[sidx][hq][e] + om[sidx][hq], k * C + c);
            ov[e] += wb[sidx][e] * x;
          }
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
        merge_unit<__nv_bfloat16, D, G>(p.ws, static_cast<__nv_bfloat16*>(p.out), u, wf, wl, N,
                                        total, b, h, H, lane);
      }
    }
  }
}

template <int D, int NSRC>
size_t q4_smem_bytes(int B) {
  using S = Q4Shape<NSRC>;
  return (size_t)S::W * S::NS * Q4Cfg<D, NSRC>::STAGE_BYTES + decode_aux_bytes(S::W, S::NS, B);
}

template <int D, int NSRC, bool WGT, int G>
cudaError_t launch_q4(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
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
  sp.counters = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(a.workspace) +
                                                      plan.partial_bytes);
  sp.status = a.status;
  sp.wait_limit = a.wait_limit;
  sp.epoch = a.epoch;
  sp.B = a.batch;
  sp.H_kv = a.kv_heads;
  sp.S_max = a.max_seq;
  sp.window = a.window;
  sp.ring = a.ring;
  sp.qscale = a.softmax_scale * 1.4426950408889634f;
  auto kern = decode_q4_kernel<D, NSRC, WGT || NSRC == 2, G>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem_bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(plan.ctas), dim3(Q4Shape<NSRC>::W * 32), plan.smem_bytes, stream, sp);
}

template <int D, int NSRC, bool WGT>
cudaError_t q4_by_group(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  switch (a.group) {
    case 1: return launch_q4<D, NSRC, WGT, 1>(a, pl, s);
    case 2: return launch_q4<D, NSRC, WGT, 2>(a, pl, s);
    default: return cudaErrorNotSupported;
  }
}

template <int D>
cudaError_t q4_by_src(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  if (a.nsrc == 2) return q4_by_group<D, 2, true>(a, pl, s);
  return a.a[0] ? q4_by_group<D, 1, true>(a, pl, s) : q4_by_group<D, 1, false>(a, pl, s);
}

}  // namespace

cudaError_t decode_q4_plan(const DecodeArgs& a, int num_sms, DecodePlan* plan) {
  if (a.is_f32 || a.group > 2) return cudaErrorNotSupported;
  size_t smem = 0;
  switch (a.head_dim) {
    case 64: smem = a.nsrc == 2 ? q4_smem_bytes<64, 2>(a.batch) : q4_smem_bytes<64, 1>(a.batch); break;
    case 80: smem = a.nsrc == 2 ? q4_smem_bytes<80, 2>(a.batch) : q4_smem_bytes<80, 1>(a.batch); break;
    case 96: smem = a.nsrc == 2 ? q4_smem_bytes<96, 2>(a.batch) : q4_smem_bytes<96, 1>(a.batch); break;
    case 128: smem = a.nsrc == 2 ? q4_smem_bytes<128, 2>(a.batch) : q4_smem_bytes<128, 1>(a.batch); break;
    default: return cudaErrorNotSupported;
  }
  const long long rows = (long long)a.batch * a.kv_heads * a.max_seq;
  long long ctas = a.num_ctas > 0 ? a.num_ctas : num_sms;
  const int W = a.nsrc == 2 ? Q4Shape<2>::W : Q4Shape<1>::W;
  const long long by_rows = (rows + 64LL * W - 1) / (64LL * W);
  if (a.num_ctas <= 0) ctas = ctas < by_rows ? ctas : by_rows;
  if (ctas < 1) ctas = 1;
  plan->ctas = (int)ctas;
  plan->warps_per_cta = W;
  plan->smem_bytes = smem;
  const size_t units = (size_t)a.batch * a.kv_heads;
  const size_t slots = (size_t)ctas * W + units;
  plan->partial_bytes = (slots * a.group * partial_stride(a.head_dim) * sizeof(float) + 15) / 16 * 16;
  plan->workspace_bytes = plan->partial_bytes + units * sizeof(unsigned long long);
  return cudaSuccess;
}

cudaError_t decode_q4_launch(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64: return q4_by_src<64>(a, plan, stream);
    case 80: return q4_by_src<80>(a, plan, stream);
    case 96: return q4_by_src<96>(a, plan, stream);
    case 128: return q4_by_src<128>(a, plan, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fkv
