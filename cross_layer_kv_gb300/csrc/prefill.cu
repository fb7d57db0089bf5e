// Causal prefill attention for FusedKV upper layers with D = 128, on the
// 5th-generation tensor cores of sm_103a, and the prefill entry point that
// picks a kernel per call (one source: prefill_wide.cu; two sources with
// D <= 96: prefill_fused_wide.cu).
//
// What one call computes: for every sequence b, query head h (KV head
// kh = h / G) and query position m < S
//     o_{h,m} = sum_{t <= m} softmax_t(scale * q_{h,m} . K_t) V_t
// with K = a_1 (.) K^1 + a_n (.) K^n and V = b_1 (.) V^1 + b_n (.) V^n (FusedKV
// slides Eqs.(4)-(5)), built tile by tile in shared memory and never written
// to global memory (Table 1 slide: fuse on demand).
//
// Structure of one CTA: one 128-row query tile of one (b, kh) unit and all G
// query heads of that KV head, with warps specialised by role:
//  * a TMA producer warp (cp.async.bulk.tensor, 64-byte swizzle) loads the Q
//    tiles once and the source tiles of 64 keys into two rings: the first
//    source's K and V (the fused tiles are written over them) and the
//    second source's;
//  * a fusion warpgroup combines the two sources of each K and V tile and
//    writes the bf16 result in place, in the swizzled layout the tensor
//    cores read (the fused tile serves all G heads); it computes in packed
//    bf16 arithmetic with each fp32 weight split as bf16 hi + lo (four packed
//    FMAs a channel pair, lo terms first);
//  * one MMA warp per head issues tcgen05.mma: S_h = Q_h K^T into a
//    double-buffered tensor-memory tile, and O_h += P_h V accumulated in
//    tensor memory; the S of the next tile is issued before the P of this one
//    is awaited, so the tensor cores work while the softmax warps run;
//  * one softmax warpgroup per head: each thread owns one query row (one TMEM
//    lane), reads its S row with tcgen05.ld, applies the causal mask and the
//    online (base-2) softmax and writes P_h (bf16) back over that S tile with
//    tcgen05.st; the PV product takes its A operand from tensor memory, so P
//    never touches shared memory;
//    O is rescaled in tensor memory only when the running max grows by more
//    than 2^8.
//  * Every wait is bounded; a wait that runs out sets an abort flag that
//    every role checks, flags the device status, and the CTA releases its
//    tensor memory and returns.
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>

#include "fkv_kernels.h"
#include "tc_device.cuh"

namespace fkv {
namespace {

constexpr int BM = 128;       // query rows per CTA
constexpr int BN = 64;        // keys per tile
constexpr int SW = kSW;       // swizzle span in bytes (32 bf16)
constexpr int SWE = kSWE;     // elements per swizzle row
constexpr int TMEM_COLS = 512;
constexpr int HEAD_COLS = 256;  // TMEM columns per head: S (BN) then O (D)

template <int D>
struct PrefillCfg {
  static constexpr int CB = (D + SWE - 1) / SWE;    // 32-element column blocks
  static constexpr int Q_BYTES = CB * BM * SW;      // one head's Q tile
  static constexpr int KV_BYTES = CB * BN * SW;     // one K or V source tile
};

struct PrefillParams {
  const float* a0;
  const float* a1;
  const float* b0;
  const float* b1;
  void* out;
  int* status;
  const unsigned long long* wait_limit;  // limit of the bounded waits (device word)
  int B, H_kv;
  int S;        // query rows of this call (the chunk length C)
  int q_start;  // cache position of the first query row
  int S_kv;     // key rows attended: q_start + C
  int window;   // > 0: a query at position m sees only keys t > m - window
  float scale_log2;
  int ring;     // > 0: K/V rows are rings of that many rows (a multiple of BN)
};

struct PrefillMaps {
  CUtensorMap q;
  CUtensorMap k0, k1, v0, v1;
};

constexpr int SMEM_LIMIT = 232448;   // opt-in dynamic shared memory per CTA (227 KB)
constexpr int AUX_BYTES = 512;       // barriers, TMEM slot, abort flag
constexpr float RESCALE_SLACK = 8.f; // log2 growth of the running max tolerated before O is rescaled

__device__ __forceinline__ __nv_bfloat162 bf162_of(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
__device__ __forceinline__ uint32_t u32_of(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D, int NSRC, int G>
struct PrefillPlan {
  using Cfg = PrefillCfg<D>;
  static_assert(NSRC == 2, "one source runs the 128-key kernel");
  // Two rings of 64-key slots: A holds the first source's K and V tile (the
  // fused tiles are written over them, and the MMA commits free a slot), B
  // the second source's (freed by the fusion warpgroup once it has read
  // them, a period or more earlier)
  static constexpr int SLOT = 2 * Cfg::KV_BYTES;
  static constexpr int FIXED = G * Cfg::Q_BYTES + 4 * D * 4 + AUX_BYTES + 512;
  static constexpr int SLOTS_FIT = (SMEM_LIMIT - FIXED) / SLOT;
  static constexpr int NB = SLOTS_FIT / 2 > 4 ? 4 : SLOTS_FIT / 2;
  static constexpr int NA = SLOTS_FIT - NB > 4 ? 4 : SLOTS_FIT - NB;
  static constexpr int SOFTMAX_WARPS = 4 * G;
  static constexpr int FUSION_WARPS = NSRC == 2 ? 4 : 0;
  static constexpr int PRODUCER_WARP = SOFTMAX_WARPS + FUSION_WARPS;
  // one MMA-issuing warp per head: a thread's mbarrier wait right after its
  // MMAs lets the tensor pipe run dry, and the other head's products fill it
  static constexpr int MMA_WARP = PRODUCER_WARP + 1;   // + h for head h
  // Two heads: 15 warps would cap every thread at 128 registers (four warps
  // on a scheduler).  An idle warp completes the producer/MMA warpgroup, and
  // register reallocation moves registers from it and the fusion warpgroup
  // to the softmax warpgroups: 2 * 128 * 168 + 128 * 104 + 128 * 56 <= 512 * 128.
  static constexpr bool SPLIT = NSRC == 2 && G == 2;
  static constexpr int THREADS = 32 * (MMA_WARP + G + (SPLIT ? 1 : 0));
  static constexpr int REGS_SOFTMAX = 168, REGS_FUSION = 104, REGS_CONTROL = 56;
  static constexpr long long REGS_SPLIT = 4LL * G * 32 * REGS_SOFTMAX + 128LL * REGS_FUSION +
                                          128LL * REGS_CONTROL;
  static_assert(!SPLIT || (THREADS == 512 && REGS_SPLIT <= 512LL * 128),
                "register split above the launch allocation");
  static_assert(NA >= 2 && NB >= 2, "shared memory too small for two slots per ring");
};

template <int D, int NSRC, int G>
size_t prefill_smem_bytes() {
  using P = PrefillPlan<D, NSRC, G>;
  size_t s = (size_t)P::FIXED + (size_t)(P::NA + P::NB) * P::SLOT;
  // at least 116 KB so that one CTA holds an SM (it takes all 512 TMEM columns)
  return s < 118784 ? 118784 : s;
}

// Warp-specialised CTA (G query heads of one KV head, 128 query rows each):
//   softmax warpgroups (one per head) | fusion warpgroup (fused mode) |
//   TMA producer warp | one MMA warp per head.
// Pipeline per 64-key tile j, all hand-offs through mbarriers:
//   producer:  a_empty -> TMA first-source K/V -> a_full;
//              b_empty -> TMA second-source K/V -> b_full
//   fusion:    a_full, b_full -> fused bf16 K/V written over the first
//              source's tiles -> b_empty, kv_ready
//   MMA of h:  kv_ready -> S_h[j%2] = Q_h K^T -> s_full[h][j%2];
//              p_full[h] -> O_h += P_h V -> o_done[h], a_empty
//              (one issuing warp per head; S of tile j+1 is issued before
//              waiting for P of tile j)
//   softmax h: s_full -> row max / exp -> (o_done of tile j-1) -> rescale O
//              in TMEM if the max grew by more than 2^8 -> P_h -> p_full[h]
template <int D, int NSRC, int G>
__global__ void __launch_bounds__(PrefillPlan<D, NSRC, G>::THREADS, 1)
    prefill_kernel(const __grid_constant__ PrefillMaps maps, const PrefillParams p) {
  using Cfg = PrefillCfg<D>;
  using PL = PrefillPlan<D, NSRC, G>;
  constexpr int CB = Cfg::CB, NA = PL::NA, NB = PL::NB;
  extern __shared__ uint8_t smem_raw[];
  // 512-byte alignment: the period of the 64-byte swizzle pattern
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) &
                                             ~uintptr_t(511));
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + G * Cfg::Q_BYTES;
  uint8_t* sB = sKV + NA * PL::SLOT;
  // the fusion weights a0, a1, b0, b1, each as D/2 bf16 pairs split in two:
  // w = hi + lo, hi = bf16(w), lo = bf16(w - hi) (hi pairs, then lo pairs)
  uint32_t* sW = reinterpret_cast<uint32_t*>(sB + NB * PL::SLOT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + 4 * D);
  uint64_t* bar_q = bars;
  uint64_t* a_full = bars + 1;          // [NA] first-source tiles landed
  uint64_t* kv_ready = a_full + NA;     // [NA] fused tiles in place
  uint64_t* a_empty = kv_ready + NA;    // [NA] MMA done with the slot
  uint64_t* b_full = a_empty + NA;      // [NB] second-source tiles landed
  uint64_t* b_empty = b_full + NB;      // [NB] fusion done with the slot
  uint64_t* s_full = b_empty + NB;      // [G][2]
  uint64_t* p_full = s_full + 2 * G;    // [G]
  uint64_t* o_done = p_full + G;        // [G]
  uint64_t* mma_drain = o_done + G;     // [G] an issuer's last products, after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + G);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* sm_issued = reinterpret_cast<int*>(tmem_slot + 2);   // copies the producer issued

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int unit, mt;
  prefill_cta_tile(unit, mt);   // longest query tiles first
  const int b = unit / p.H_kv, kh = unit % p.H_kv;
  const int m0 = mt * BM;              // first query row of the tile (within the chunk)
  const int S = p.S;                   // query rows
  const int S_kv = p.S_kv;             // key rows
  const int pos0 = p.q_start + m0;     // cache position of query row m0
  const int W = p.window;
  // key tiles [j0, j_end): up to the last query's position, from the first
  // query's window start (sliding-window layers skip the tiles before it)
  const int j0 = W > 0 ? max(0, pos0 - W + 1) / BN : 0;
  const int ntiles = (min(pos0 + BM, S_kv) + BN - 1) / BN - j0;   // tiles processed
  const int H_q = p.H_kv * G;
  const unsigned long long wlim = wait_limit_ns(p.wait_limit);

  // key tile j: source src's K or V tile
  auto stage_k = [&](int j, int src) {
    return src == 0 ? sKV + (size_t)(j % NA) * PL::SLOT : sB + (size_t)(j % NB) * PL::SLOT;
  };
  auto stage_v = [&](int j, int src) { return stage_k(j, src) + Cfg::KV_BYTES; };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, wlim)) return true;
    *abort_flag = 1;
    flag_status(p.status, kDevTimeout);
    return false;
  };

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&kv_ready[s], 128);
      mbar_init(&a_empty[s], G);   // one commit per head's issuer
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 128);
    }
    for (int h = 0; h < G; ++h) {
      mbar_init(&s_full[2 * h], 1);
      mbar_init(&s_full[2 * h + 1], 1);
      mbar_init(&p_full[h], 128);
      mbar_init(&o_done[h], 1);
      mbar_init(&mma_drain[h], 1);
    }
    *abort_flag = 0;
    *sm_issued = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * D; i += PL::THREADS) {   // (vector, channel pair)
    const int v = i / (D / 2), pc = i % (D / 2);
    const float* src = v == 0 ? p.a0 : v == 1 ? p.a1 : v == 2 ? p.b0 : p.b1;
    const float w0 = src[kh * D + 2 * pc], w1 = src[kh * D + 2 * pc + 1];
    const __nv_bfloat162 hi = __floats2bfloat162_rn(w0, w1);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(w0 - __low2float(hi), w1 - __high2float(hi));
    sW[v * D + pc] = *reinterpret_cast<const uint32_t*>(&hi);
    sW[v * D + D / 2 + pc] = *reinterpret_cast<const uint32_t*>(&lo);
  }
  if (warp == PL::MMA_WARP) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if constexpr (PL::SPLIT) {
    if (warp >= PL::PRODUCER_WARP)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PL::REGS_CONTROL));
  }
  if (warp == PL::PRODUCER_WARP) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, G * Cfg::Q_BYTES);
      for (int h = 0; h < G; ++h)
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(sQ + h * Cfg::Q_BYTES + cb * BM * SW, &maps.q, cb * SWE, m0,
                      b * H_q + kh * G + h, bar_q);
      int issued = 0;   // copies issued: 2 per tile (ring A, then ring B)
      for (int j = 0; j < ntiles; ++j) {
        const int n0 = (j0 + j) * BN;
        // the tile's first cache row: in a ring, whole tiles never wrap
        const int ky = p.ring > 0 ? n0 % p.ring : n0;
        if (j >= NA && !wait(&a_empty[j % NA], (uint32_t)(j / NA - 1) & 1u)) break;
        mbar_arrive_expect_tx(&a_full[j % NA], PL::SLOT);
        for (int cb = 0; cb < CB; ++cb) {
          tma_load_3d(stage_k(j, 0) + cb * BN * SW, &maps.k0, cb * SWE, ky, unit, &a_full[j % NA]);
          tma_load_3d(stage_v(j, 0) + cb * BN * SW, &maps.v0, cb * SWE, ky, unit, &a_full[j % NA]);
        }
        issued = 2 * j + 1;
        if (j >= NB && !wait(&b_empty[j % NB], (uint32_t)(j / NB - 1) & 1u)) break;
        mbar_arrive_expect_tx(&b_full[j % NB], PL::SLOT);
        for (int cb = 0; cb < CB; ++cb) {
          tma_load_3d(stage_k(j, 1) + cb * BN * SW, &maps.k1, cb * SWE, ky, unit, &b_full[j % NB]);
          tma_load_3d(stage_v(j, 1) + cb * BN * SW, &maps.v1, cb * SWE, ky, unit, &b_full[j % NB]);
        }
        issued = 2 * j + 2;
      }
      *sm_issued = issued;
    }
  } else if (warp >= PL::MMA_WARP && warp < PL::MMA_WARP + G) {
    // ---------------- MMA issuer of head h ----------------
    const int h = warp - PL::MMA_WARP;
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, true);
      const uint32_t qbase = smem_u32(sQ + h * Cfg::Q_BYTES);
      auto issue_qk = [&](int j) {
        const uint32_t kbase = smem_u32(stage_k(j, 0));
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k & 1) * 32;
          const uint64_t ad = sdesc(qbase + (k >> 1) * BM * SW + off, 16, 8 * SW);
          const uint64_t bd = sdesc(kbase + (k >> 1) * BN * SW + off, 16, 8 * SW);
          mma_bf16(tmem + h * HEAD_COLS + (j & 1) * BN, ad, bd, IDESC_QK, k > 0);
        }
        mma_commit(&s_full[2 * h + (j & 1)]);
      };
      bool ok = wait(bar_q, 0) && wait(&kv_ready[0], 0);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        // S of tile j+1 goes to the other S buffer before P of tile j is awaited
        if (j + 1 < ntiles) {
          if (!wait(&kv_ready[(j + 1) % NA], (uint32_t)((j + 1) / NA) & 1u)) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        if (!wait(&p_full[h], (uint32_t)j & 1u)) break;
        tc_fence_after();
        // P_h (bf16, two per column) sits in the first BN/2 columns of the
        // S tile it was computed from
        const uint32_t vbase = smem_u32(stage_v(j, 0));
        const uint32_t ptmem = tmem + h * HEAD_COLS + (j & 1) * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = sdesc(vbase + k * 16 * SW, BN * SW, 8 * SW);
          mma_bf16_ts(tmem + h * HEAD_COLS + 2 * BN, ptmem + k * 8, bd, IDESC_PV,
                      (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&o_done[h]);
        mma_commit(&a_empty[j % NA]);
      }
    }
  } else if (warp >= PL::SOFTMAX_WARPS && warp < PL::PRODUCER_WARP) {
    // ---------------- fusion warpgroup (fused mode) ----------------
    if constexpr (NSRC == 2) {
      if constexpr (PL::SPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PL::REGS_FUSION));
      const int ft = tid - 32 * PL::SOFTMAX_WARPS;   // 0..127
      // The thread's 16-byte chunks of a source tile are ft + 128 i: chunk i
      // lies in column block i / 2 (a block holds BN rows of 4 chunks) and,
      // the swizzle term being ((row >> 1) & 3) with row = ft / 4 + 32 i
      // mod BN, always at the same logical chunk of its row.  So the thread
      // needs the weights of one 8-column group per column block.
      static_assert(BN * 4 == 256, "two chunks of a thread per column block");
      const int lc = (ft & 3) ^ ((ft >> 3) & 3);
      for (int j = 0; j < ntiles; ++j) {
        if (!wait(&a_full[j % NA], (uint32_t)(j / NA) & 1u) ||
            !wait(&b_full[j % NB], (uint32_t)(j / NB) & 1u))
          break;
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          uint8_t* d0 = t == 0 ? stage_k(j, 0) : stage_v(j, 0);
          const uint8_t* d1 = t == 0 ? stage_k(j, 1) : stage_v(j, 1);
          const uint32_t* w0 = sW + (t == 0 ? 0 : 2 * D);
          const uint32_t* w1 = sW + (t == 0 ? D : 3 * D);
          // all of the thread's chunks of both sources first, so that no
          // load waits behind the stores of an earlier chunk
          constexpr int PER = 2 * CB;
          uint4 xs[PER], ys[PER];
#pragma unroll
          for (int i = 0; i < PER; ++i) {
            const int c = ft + 128 * i;
            xs[i] = *reinterpret_cast<const uint4*>(d0 + (size_t)c * 16);
            ys[i] = *reinterpret_cast<const uint4*>(d1 + (size_t)c * 16);
          }
#pragma unroll
          for (int cb = 0; cb < CB; ++cb) {
            const int col = cb * SWE + lc * 8;
            if (col >= D) continue;  // padding columns stay zero
            // the block's 4 weight pairs of each source, hi and lo: 16 bytes apiece
            const int pc = col / 2;
            const uint4 h0 = *reinterpret_cast<const uint4*>(w0 + pc);
            const uint4 l0 = *reinterpret_cast<const uint4*>(w0 + D / 2 + pc);
            const uint4 h1 = *reinterpret_cast<const uint4*>(w1 + pc);
            const uint4 l1 = *reinterpret_cast<const uint4*>(w1 + D / 2 + pc);
            const uint32_t w0h[4] = {h0.x, h0.y, h0.z, h0.w}, w0l[4] = {l0.x, l0.y, l0.z, l0.w};
            const uint32_t w1h[4] = {h1.x, h1.y, h1.z, h1.w}, w1l[4] = {l1.x, l1.y, l1.z, l1.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int i = 2 * cb + h;
              const uint4 x = xs[i], y = ys[i];
              const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // a0 * x + a1 * y per channel pair in packed bf16 arithmetic,
                // each weight as hi + lo (lo products first; one rounding of
                // the a1 * y partial sum and the final one)
                const __nv_bfloat162 xb = bf162_of(xw[e]), yb = bf162_of(yw[e]);
                __nv_bfloat162 acc = __hmul2(bf162_of(w0l[e]), xb);
                acc = __hfma2(bf162_of(w1l[e]), yb, acc);
                acc = __hfma2(bf162_of(w1h[e]), yb, acc);
                acc = __hfma2(bf162_of(w0h[e]), xb, acc);
                o[e] = u32_of(acc);
              }
              *reinterpret_cast<uint4*>(d0 + (size_t)(ft + 128 * i) * 16) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
        mbar_arrive(&b_empty[j % NB]);   // the second source's tiles are read
        fence_proxy_async_smem();
        mbar_arrive(&kv_ready[j % NA]);
      }
    }
  } else if (warp < PL::SOFTMAX_WARPS) {
    // ---------------- softmax warpgroup of head hh ----------------
    if constexpr (PL::SPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PL::REGS_SOFTMAX));
    const int hh = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qpos = pos0 + row;         // cache position of this query
    const bool row_valid = m0 + row < S;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_head = tmem + lane_addr + hh * HEAD_COLS;
    const uint32_t t_o = t_head + 2 * BN;
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int n0 = (j0 + j) * BN;
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, wait(&s_full[2 * hh + (j & 1)], (uint32_t)(j >> 1) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c = 0; c < BN; c += 16) tmem_ld16(t_head + (j & 1) * BN + c, sv + c);
      tmem_wait_ld();
      // masking needed: the causal diagonal, the key extent, or (window) the
      // lowest row-window start of the tile (warp-uniform)
      const bool diag = n0 + BN > pos0 || n0 + BN > S_kv || (W > 0 && n0 < pos0 + BM - W);
      if (diag) {
        const int lo = W > 0 ? qpos - W + 1 : INT_MIN;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int kp = n0 + c;
          if (kp > qpos || kp >= S_kv || kp < lo) sv[c] = -INFINITY;
        }
      }
      // row max of the raw scores (the scale is positive, so it commutes)
      float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx0 = fmaxf(mx0, sv[c]);
        mx1 = fmaxf(mx1, sv[c + 1]);
        mx2 = fmaxf(mx2, sv[c + 2]);
        mx3 = fmaxf(mx3, sv[c + 3]);
      }
      const float mt_row = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
      // Keep a stale max until it is exceeded by more than 2^8: P stays
      // below 256 (exact in bf16 and fp32) and O needs no rescaling.
      const float m_new = mt_row > m_run + RESCALE_SLACK ? mt_row : m_run;
      const float alpha = fast_exp2(m_run - m_new);
      const float neg_m = -m_new;
      float ps0 = 0.f, ps1 = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        // x = s * scale - m for two scores with one packed FMA; exp2(-inf) = 0
        float x0 = neg_m, x1 = neg_m;
        fma2(x0, x1, sv[c], sv[c + 1], p.scale_log2, p.scale_log2);
        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
        add2(ps0, ps1, e0, e1);
        __nv_bfloat162 v2 = __floats2bfloat162_rn(e0, e1);
        pk[c / 2] = *reinterpret_cast<uint32_t*>(&v2);
      }
      const float psum = ps0 + ps1;
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (j > 0) {
        // PV of tile j-1 must be done: it reads P_h and accumulates O_h
        if (!__all_sync(0xffffffffu, wait(&o_done[hh], (uint32_t)(j - 1) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
          for (int c = 0; c < D; c += 16) {
            float ov[16];
            tmem_ld16(t_o + c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= alpha;
            tmem_st16(t_o + c, ov);
          }
          tmem_wait_st();
        }
      }
      // P over the S tile just read (its first BN/2 columns): the MMA reads it
      // from tensor memory as the A operand of O += P V
      static_assert(BN / 2 == 32, "one 32-column store per row");
      tmem_st32(t_head + (j & 1) * BN, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[hh]);
    }
    if (ok && __all_sync(0xffffffffu, wait(&o_done[hh], (uint32_t)(ntiles - 1) & 1u))) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            (((size_t)b * H_q + kh * G + hh) * S + m0 + row) * D;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float ov[16];
        tmem_ld16(t_o + c, ov);
        tmem_wait_ld();
        uint32_t q8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          __nv_bfloat162 v2 = __floats2bfloat162_rn(ov[2 * e] * inv, ov[2 * e + 1] * inv);
          q8[e] = *reinterpret_cast<uint32_t*>(&v2);
        }
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
          dst[0] = make_uint4(q8[0], q8[1], q8[2], q8[3]);
          dst[1] = make_uint4(q8[4], q8[5], q8[6], q8[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out somewhere, so no role may have awaited the last copies
    // and products: the producer lets its copies in flight land (Q and the
    // last tiles of each ring; an older tile was consumed before its slot was
    // refilled) and each issuer lets its own products finish, before the CTA
    // frees tensor memory and exits.
    if (warp == PL::PRODUCER_WARP && lane == 0) {
      (void)mbar_wait_bounded(bar_q, 0, kDrainLimitNs);
      const int issued = *sm_issued;
      const int ta = (issued + 1) / 2, tb = issued / 2;   // tiles issued per ring
      for (int j = max(0, ta - NA); j < ta; ++j)
        (void)mbar_wait_bounded(&a_full[j % NA], (uint32_t)(j / NA) & 1u, kDrainLimitNs);
      for (int j = max(0, tb - NB); j < tb; ++j)
        (void)mbar_wait_bounded(&b_full[j % NB], (uint32_t)(j / NB) & 1u, kDrainLimitNs);
    }
    if (warp >= PL::MMA_WARP && warp < PL::MMA_WARP + G && lane == 0) {
      mma_commit(&mma_drain[warp - PL::MMA_WARP]);
      (void)mbar_wait_bounded(&mma_drain[warp - PL::MMA_WARP], 0, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == PL::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// --- host side ---------------------------------------------------------------

template <int D, int NSRC, int G>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t stream) {
  PrefillMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const long long units = (long long)a.batch * a.kv_heads;
  const size_t kv_plane = (size_t)a.plane_rows * D * 2;   // bytes per (b, kv-head) plane
  const int S_kv = a.q_start + a.S;
  // a ring whose positions have wrapped is read whole (rows past the key
  // extent hold older positions, masked); otherwise rows from S_kv on read 0.
  // Whole key tiles map to whole ring rows only if the ring is a multiple of BN.
  const bool wrapped = a.ring > 0 && S_kv > a.ring;
  if (wrapped && a.ring % BN != 0) return cudaErrorNotSupported;
  const int map_rows = wrapped ? a.ring : S_kv;
  bool ok = make_map(&maps.q, a.q, D, a.S, (long long)a.batch * a.kv_heads * G,
                     (size_t)a.S * D * 2, BM);
  ok = ok && make_map(&maps.k0, a.k[0], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.v0, a.v[0], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.k1, a.k[1], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.v1, a.v[1], D, map_rows, units, kv_plane, BN);
  if (!ok) return cudaErrorInvalidValue;
  PrefillParams p;
  p.a0 = a.a[0];
  p.a1 = a.a[1];
  p.b0 = a.b[0];
  p.b1 = a.b[1];
  p.out = a.out;
  p.status = a.status;
  p.wait_limit = a.wait_limit;
  p.B = a.batch;
  p.H_kv = a.kv_heads;
  p.S = a.S;
  p.q_start = a.q_start;
  p.S_kv = S_kv;
  p.window = a.window;
  p.ring = a.ring;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  const size_t smem = prefill_smem_bytes<D, NSRC, G>();
  auto kern = prefill_kernel<D, NSRC, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (PrefillPlan<D, NSRC, G>::SPLIT) {
    // the softmax warpgroups' register increase must fit the launch
    // allocation, or it would never be granted: refuse instead
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if ((long long)fa.numRegs * PrefillPlan<D, NSRC, G>::THREADS < PrefillPlan<D, NSRC, G>::REGS_SPLIT)
      return cudaErrorNotSupported;
  }
  dim3 grid((unsigned)units, (unsigned)((a.S + BM - 1) / BM));
  kern<<<grid, PrefillPlan<D, NSRC, G>::THREADS, smem, stream>>>(maps, p);
  return cudaGetLastError();
}

// two sources (fused); one source goes to the 128-key kernel
template <int D>
cudaError_t by_group(const PrefillArgs& a, cudaStream_t s) {
  if (a.group == 1) return launch_t<D, 2, 1>(a, s);
  if (a.group == 2) return launch_t<D, 2, 2>(a, s);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t prefill_launch(const PrefillArgs& a, cudaStream_t stream) {
  if (a.batch * (long long)a.kv_heads > 65535 || a.S < 1) return cudaErrorNotSupported;
  if (a.nsrc == 1) return prefill_wide_launch(a, stream);
  if (a.nsrc != 2) return cudaErrorNotSupported;
  if (a.head_dim <= 96) return prefill_fused_wide_launch(a, stream);
  if (a.head_dim == 128) return by_group<128>(a, stream);
  return cudaErrorNotSupported;
}

}  // namespace fkv
