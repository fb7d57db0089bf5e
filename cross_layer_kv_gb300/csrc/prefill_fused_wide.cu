// Causal prefill attention for FusedKV upper layers whose keys and values are
// rebuilt from two stored layers, K = a_1 (.) K^1 + a_n (.) K^n and
// V = b_1 (.) V^1 + b_n (.) V^n (FusedKV slides Eqs.(4)-(5)), tile by tile in
// shared memory and never written to global memory (Table 1 slide: fuse on
// demand), on the tcgen05 tensor cores of sm_103a with 112-key tiles.
//
// What one call computes: for every sequence b, query head h (KV head
// kh = h / G) and query position m of the chunk
//     o_{h,m} = sum_{t <= m, t > m - W} softmax_t(scale * q_{h,m} . K_t) V_t.
//
// Design.  As in the one-source kernel (prefill_wide.cu), a CTA owns two
// groups of 128 query rows that read the same keys (the two heads of one KV
// head, or two row tiles of one head), each with a softmax warpgroup and one
// MMA-issuing warp, and the issuers take turns on the tensor pipe.  What
// differs is where the operands live:
//  * Q sits in tensor memory.  Each group's 256 columns hold S_g / P_g
//    (112 fp32 columns), O_g (D columns) and Q_g (D/2 packed bf16 columns),
//    so S_g = Q_g K^T reads A from tensor memory and K from shared memory,
//    and shared memory is left to the source tiles.
//  * Four rings of 112-key tiles: the first source's K and V (the fused
//    tiles are written over them and the MMA commits free a slot) and the
//    second source's K and V (freed by the fusion warpgroup as soon as it has
//    read them).
//  * A fusion warpgroup combines the two sources of each tile and writes
//    bf16 over the first source's tile, in the swizzled layout the MMA reads.
//    It computes in packed bf16 arithmetic (two channels an instruction),
//    each fp32 weight split as bf16 hi + lo so that no weight is rounded:
//    four packed FMAs a channel pair instead of seven fp32 operations with
//    their conversions, at the cost of one rounding of the second source's
//    partial product.  Its step k fuses V_{k-1} and K_k, the tiles MMA step
//    k reads, and signals one barrier per step.
// Every wait is bounded; a wait that runs out sets an abort flag that each
// role checks, flags the device status, and the CTA frees its tensor memory.
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>

#include "fkv_kernels.h"
#include "tc_device.cuh"

namespace fkv {
namespace {

constexpr int BM = 128;          // query rows per group
constexpr int BN = 112;          // keys per tile
constexpr int NG = 2;            // groups per CTA
constexpr int GROUP_COLS = 256;  // TMEM columns per group: S/P, O, Q
constexpr int SW = kSW;
constexpr int SWE = kSWE;
constexpr int SMEM_LIMIT = 232448;   // opt-in dynamic shared memory per CTA (227 KB)
constexpr float RESCALE_SLACK = 8.f; // log2 growth of the running max tolerated before O is rescaled
constexpr int NSR = 8;               // fusion-step barriers (more than any ring has slots)

constexpr int cap4(int x) { return x > 4 ? 4 : x; }

__device__ __forceinline__ __nv_bfloat162 bf162_of(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
__device__ __forceinline__ uint32_t u32_of(__nv_bfloat162 v) {
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
struct FwCfg {
  static constexpr int CB = (D + SWE - 1) / SWE;      // 32-element column blocks
  static constexpr int KV_BYTES = CB * BN * SW;       // one K or V tile of one source
  static constexpr int O_COL = BN;                    // O_g: columns [BN, BN + D)
  static constexpr int Q_COLS = (D / 2 + 15) / 16 * 16;
  static constexpr int Q_COL = GROUP_COLS - Q_COLS;   // Q_g: D/2 packed bf16 columns
  static_assert(O_COL + D <= Q_COL, "S, O and Q do not fit a group's 256 columns");
  static constexpr int FIXED = 4 * D * 4 + 1024;      // weights, barriers
  static constexpr int TILES_FIT = (SMEM_LIMIT - 512 - FIXED) / KV_BYTES;
  // first-source rings of NSK slots (3 at D = 96), second-source rings of NS1 (2)
  static constexpr int NSK = cap4((TILES_FIT - 4) / 2);
  static constexpr int NSV = NSK;
  static constexpr int NS1 = cap4((TILES_FIT - NSK - NSV) / 2);
  static_assert(NSK >= 2 && NS1 >= 2, "shared memory too small for the fused rings");
  static_assert(NSR > NSK && NSR > NSV, "step barriers must outnumber the ring slots");
  static constexpr size_t SMEM = 512 + (size_t)FIXED + (size_t)(NSK + NSV + 2 * NS1) * KV_BYTES;
  static_assert(SMEM <= SMEM_LIMIT, "shared memory above the opt-in limit");
  static constexpr int SOFTMAX_WARPS = 4 * NG;
  static constexpr int K_PRODUCER_WARP = SOFTMAX_WARPS;
  static constexpr int MMA_WARP = K_PRODUCER_WARP + 1;   // + g for group g
  static constexpr int V_PRODUCER_WARP = MMA_WARP + NG;
  static constexpr int FUSION_WARP = SOFTMAX_WARPS + 4;
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 8);
  // registers: 128 per thread at launch (65536 / 512); the control and
  // fusion warpgroups give some up and the softmax warpgroups take them
#ifdef FKV_PFW_REGS_CONTROL
  static constexpr int REGS_CONTROL = FKV_PFW_REGS_CONTROL;   // tuning sweeps
  static constexpr int REGS_FUSION = FKV_PFW_REGS_FUSION;
  static constexpr int REGS_SOFTMAX = FKV_PFW_REGS_SOFTMAX;
#else
  static constexpr int REGS_CONTROL = 56, REGS_FUSION = 80, REGS_SOFTMAX = 184;
#endif
  static constexpr long long REGS_SPLIT =
      (long long)NG * 128 * REGS_SOFTMAX + 128LL * REGS_CONTROL + 128LL * REGS_FUSION;
  static_assert(REGS_SPLIT <= (long long)THREADS * 128, "register split above the launch allocation");
};

struct FwParams {
  const float* a0;   // fusion weights of the first and second source [H_kv, D]
  const float* a1;
  const float* b0;
  const float* b1;
  const void* q;     // [B, H_q, S, D] bf16
  void* out;         // [B, H_q, S, D] bf16
  int* status;
  const unsigned long long* wait_limit;  // limit of the bounded waits (device word)
  int H_kv, G;
  int S;        // query rows of this call (the chunk length C)
  int q_start;  // cache position of query row 0
  int S_kv;     // key rows attended: q_start + C
  int window;   // > 0: a query at position m sees only keys t > m - window
  float scale_log2;
  int ring;     // > 0: K/V rows are rings of that many rows (a multiple of BN)
};

struct FwMaps {
  CUtensorMap k0, k1, v0, v1;
};

template <int D>
__global__ void __launch_bounds__(FwCfg<D>::THREADS, 1)
    prefill_fused_wide_kernel(const __grid_constant__ FwMaps maps, const FwParams p) {
  using C = FwCfg<D>;
  constexpr int CB = C::CB, NSK = C::NSK, NSV = C::NSV, NS1 = C::NS1;
  extern __shared__ uint8_t smem_raw[];
  // 512-byte alignment: the period of the 64-byte swizzle pattern
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) &
                                             ~uintptr_t(511));
  uint8_t* sK = smem;                                  // first source, fused in place
  uint8_t* sV = sK + NSK * C::KV_BYTES;
  uint8_t* sK1 = sV + NSV * C::KV_BYTES;               // second source
  uint8_t* sV1 = sK1 + NS1 * C::KV_BYTES;
  // the fusion weights a0, a1, b0, b1, each as D/2 bf16 pairs split in two:
  // w = hi + lo, hi = bf16(w), lo = bf16(w - hi) (hi pairs, then lo pairs)
  uint32_t* sW = reinterpret_cast<uint32_t*>(sV1 + NS1 * C::KV_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + 4 * D);
  uint64_t* q_ready = bars;
  uint64_t* k_full = q_ready + 1;   // [4] each ring's barriers, padded to 4
  uint64_t* k_empty = k_full + 4;
  uint64_t* v_full = k_empty + 4;
  uint64_t* v_empty = v_full + 4;
  uint64_t* k1_full = v_empty + 4;
  uint64_t* k1_empty = k1_full + 4;
  uint64_t* v1_full = k1_empty + 4;
  uint64_t* v1_empty = v1_full + 4;
  uint64_t* step_ready = v1_empty + 4;   // [NSR]
  uint64_t* s_full = step_ready + NSR;   // [NG]
  uint64_t* p_full = s_full + NG;        // [NG]
  uint64_t* mma_drain = p_full + NG;     // [NG] an issuer's last products, after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + NG);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* sm_issued = reinterpret_cast<int*>(tmem_slot + 2);   // [2] copies each producer issued
  static_assert(NSK <= 4 && NSV <= 4 && NS1 <= 4, "barrier arrays hold 4 slots");

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int unit, mt;
  prefill_cta_tile(unit, mt);   // longest query tiles first
  const int H_q = p.H_kv * p.G;
  const int b = unit / p.H_kv, kh = unit % p.H_kv;
  const bool two_heads = p.G == 2;
  // group g: query head and first query row (within the chunk)
  auto g_head = [&](int g) { return two_heads ? kh * 2 + g : kh; };
  auto g_row0 = [&](int g) { return two_heads ? mt * BM : mt * (NG * BM) + g * BM; };
  const int S_kv = p.S_kv;
  const int W = p.window;
  // key tiles [j0, j0 + n_g): from the first group's window start up to each
  // group's last query position
  const int pos_first = p.q_start + g_row0(0);
  const int j0 = W > 0 ? max(0, pos_first - W + 1) / BN : 0;
  auto n_tiles = [&](int g) { return (min(p.q_start + g_row0(g) + BM, S_kv) + BN - 1) / BN - j0; };
  const int n_max = max(n_tiles(0), n_tiles(1));
  const unsigned long long wlim = wait_limit_ns(p.wait_limit);

  auto tile_k = [&](int j) { return sK + (size_t)(j % NSK) * C::KV_BYTES; };
  auto tile_v = [&](int j) { return sV + (size_t)(j % NSV) * C::KV_BYTES; };
  auto tile_k1 = [&](int j) { return sK1 + (size_t)(j % NS1) * C::KV_BYTES; };
  auto tile_v1 = [&](int j) { return sV1 + (size_t)(j % NS1) * C::KV_BYTES; };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, wlim)) return true;
    *abort_flag = 1;
    flag_status(p.status, kDevTimeout);
    return false;
  };

  if (tid == 0) {
    mbar_init(q_ready, 128 * NG);
    for (int s = 0; s < NSR; ++s) mbar_init(&step_ready[s], 128);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], NG);    // one commit per group that reads the tile
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], NG);
      mbar_init(&k1_full[s], 1);
      mbar_init(&k1_empty[s], 128);  // the fusion threads, once they have read it
      mbar_init(&v1_full[s], 1);
      mbar_init(&v1_empty[s], 128);
    }
    for (int g = 0; g < NG; ++g) {
      mbar_init(&s_full[g], 1);
      // the group's 128 softmax threads, plus the other group's issuer once
      // its previous step's PV products are queued (the turn)
      mbar_init(&p_full[g], 129);
      mbar_init(&mma_drain[g], 1);
    }
    *abort_flag = 0;
    sm_issued[0] = sm_issued[1] = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * D; i += C::THREADS) {   // (vector, channel pair)
    const int v = i / (D / 2), pc = i % (D / 2);
    const float* src = v == 0 ? p.a0 : v == 1 ? p.a1 : v == 2 ? p.b0 : p.b1;
    const float w0 = src[kh * D + 2 * pc], w1 = src[kh * D + 2 * pc + 1];
    const __nv_bfloat162 hi = __floats2bfloat162_rn(w0, w1);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(w0 - __low2float(hi), w1 - __high2float(hi));
    sW[v * D + pc] = *reinterpret_cast<const uint32_t*>(&hi);
    sW[v * D + D / 2 + pc] = *reinterpret_cast<const uint32_t*>(&lo);
  }
  if (warp == C::MMA_WARP) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::FUSION_WARP) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_FUSION));
    // ---------------- fusion warpgroup ----------------
    const int ft = tid - 32 * C::FUSION_WARP;   // 0..127
    // Within a column block (BN rows of four 16-byte chunks) the thread takes
    // chunks ft + 128 i, i.e. rows ft / 4 + 32 i, at physical chunk ft & 3;
    // the 64-byte swizzle term ((row >> 1) & 3) is then (ft >> 3) & 3 for
    // all of them, so the thread combines one 8-column group per block.
    const int lc = (ft & 3) ^ ((ft >> 3) & 3);
    constexpr int PER_BLOCK = (BN * 4 + 127) / 128;   // 4 (the last one for ft < 64)
    // w0, w1: the split weight pairs of the two sources (hi pairs at [0, D/2),
    // lo pairs at [D/2, D))
    auto fuse = [&](uint8_t* d0, const uint8_t* d1, const uint32_t* w0, const uint32_t* w1) {
#pragma unroll
      for (int cb = 0; cb < CB; ++cb) {
        const int col = cb * SWE + lc * 8;
        if (col >= D) continue;  // padding columns stay zero
        // the block's chunks of both sources first, then combine and store
        uint4 xs[PER_BLOCK], ys[PER_BLOCK];
#pragma unroll
        for (int i = 0; i < PER_BLOCK; ++i) {
          const int q = ft + 128 * i;
          if (q < BN * 4) {
            xs[i] = *reinterpret_cast<const uint4*>(d0 + (size_t)(cb * BN * 4 + q) * 16);
            ys[i] = *reinterpret_cast<const uint4*>(d1 + (size_t)(cb * BN * 4 + q) * 16);
          }
        }
        // the block's 4 weight pairs of each source, hi and lo: 16 bytes apiece
        const int pc = col / 2;
        const uint4 h0 = *reinterpret_cast<const uint4*>(w0 + pc);
        const uint4 l0 = *reinterpret_cast<const uint4*>(w0 + D / 2 + pc);
        const uint4 h1 = *reinterpret_cast<const uint4*>(w1 + pc);
        const uint4 l1 = *reinterpret_cast<const uint4*>(w1 + D / 2 + pc);
        const uint32_t w0h[4] = {h0.x, h0.y, h0.z, h0.w}, w0l[4] = {l0.x, l0.y, l0.z, l0.w};
        const uint32_t w1h[4] = {h1.x, h1.y, h1.z, h1.w}, w1l[4] = {l1.x, l1.y, l1.z, l1.w};
#pragma unroll
        for (int i = 0; i < PER_BLOCK; ++i) {
          const int q = ft + 128 * i;
          if (q >= BN * 4) continue;
          const uint32_t xw[4] = {xs[i].x, xs[i].y, xs[i].z, xs[i].w};
          const uint32_t yw[4] = {ys[i].x, ys[i].y, ys[i].z, ys[i].w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // w0 * x + w1 * y per channel pair in packed bf16 arithmetic, with
            // each weight as hi + lo so that it keeps its fp32 value to 2^-16:
            // the small lo products first, then the hi products; one rounding
            // of the w1 * y partial sum and the final one
            const __nv_bfloat162 x = bf162_of(xw[e]), y = bf162_of(yw[e]);
            __nv_bfloat162 acc = __hmul2(bf162_of(w0l[e]), x);
            acc = __hfma2(bf162_of(w1l[e]), y, acc);
            acc = __hfma2(bf162_of(w1h[e]), y, acc);
            acc = __hfma2(bf162_of(w0h[e]), x, acc);
            o[e] = u32_of(acc);
          }
          *reinterpret_cast<uint4*>(d0 + (size_t)(cb * BN * 4 + q) * 16) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    };
    // step 0 fuses K_0; step k > 0 fuses V_{k-1}, then K_k (k < n_max)
    for (int k = 0; k <= n_max; ++k) {
      if (k > 0) {
        const int t = k - 1;
        if (!wait(&v_full[t % NSV], (uint32_t)(t / NSV) & 1u) ||
            !wait(&v1_full[t % NS1], (uint32_t)(t / NS1) & 1u))
          break;
        fuse(tile_v(t), tile_v1(t), sW + 2 * D, sW + 3 * D);
        mbar_arrive(&v1_empty[t % NS1]);
      }
      if (k < n_max) {
        if (!wait(&k_full[k % NSK], (uint32_t)(k / NSK) & 1u) ||
            !wait(&k1_full[k % NS1], (uint32_t)(k / NS1) & 1u))
          break;
        fuse(tile_k(k), tile_k1(k), sW, sW + D);
        mbar_arrive(&k1_empty[k % NS1]);
      }
      // the fused tiles are read by the tensor cores (async proxy)
      fence_proxy_async_smem();
      mbar_arrive(&step_ready[k % NSR]);
    }
  } else if (warp >= C::SOFTMAX_WARPS) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CONTROL));
    if ((warp == C::K_PRODUCER_WARP || warp == C::V_PRODUCER_WARP) && lane == 0) {
      // ---------------- TMA producers: K tiles, V tiles ----------------
      // first source into its ring (freed by the MMA commits), second into
      // its own (freed by the fusion warpgroup)
      const bool is_k = warp == C::K_PRODUCER_WARP;
      const int n0s = is_k ? NSK : NSV;
      uint64_t* f0 = is_k ? k_full : v_full;
      uint64_t* e0 = is_k ? k_empty : v_empty;
      uint64_t* f1 = is_k ? k1_full : v1_full;
      uint64_t* e1 = is_k ? k1_empty : v1_empty;
      const CUtensorMap* m0 = is_k ? &maps.k0 : &maps.v0;
      const CUtensorMap* m1 = is_k ? &maps.k1 : &maps.v1;
      int issued = 0;   // copies issued: 2 per tile (first source, then second)
      for (int j = 0; j < n_max; ++j) {
        const int n0 = (j0 + j) * BN;
        // the tile's first cache row: in a ring, whole tiles never wrap
        const int ky = p.ring > 0 ? n0 % p.ring : n0;
        if (j >= n0s && !wait(&e0[j % n0s], (uint32_t)(j / n0s - 1) & 1u)) break;
        uint8_t* d0 = is_k ? tile_k(j) : tile_v(j);
        mbar_arrive_expect_tx(&f0[j % n0s], C::KV_BYTES);
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(d0 + cb * BN * SW, m0, cb * SWE, ky, unit, &f0[j % n0s]);
        issued = 2 * j + 1;
        if (j >= NS1 && !wait(&e1[j % NS1], (uint32_t)(j / NS1 - 1) & 1u)) break;
        uint8_t* d1 = is_k ? tile_k1(j) : tile_v1(j);
        mbar_arrive_expect_tx(&f1[j % NS1], C::KV_BYTES);
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(d1 + cb * BN * SW, m1, cb * SWE, ky, unit, &f1[j % NS1]);
        issued = 2 * j + 2;
      }
      sm_issued[is_k ? 0 : 1] = issued;
    } else if (warp >= C::MMA_WARP && warp < C::MMA_WARP + NG && lane == 0) {
      // ---------------- MMA issuer of group g ----------------
      const int g = warp - C::MMA_WARP;
      constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, true);
      const uint32_t t_g = tmem + g * GROUP_COLS;
      // S_g = Q_g K_j^T: A = Q_g from tensor memory (8 columns per step of 16
      // channels), B = K_j (K-major), N = 112 keys
      auto issue_qk = [&](int j) {
        const uint32_t kbase = smem_u32(tile_k(j));
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k & 1) * 32;
          const uint64_t bd = sdesc(kbase + (k >> 1) * BN * SW + off, 16, 8 * SW);
          mma_bf16_ts(t_g, t_g + C::Q_COL + k * 8, bd, IDESC_QK, k > 0);
        }
      };
      // O_g += P_g V_j: A = P_g (bf16, two per column, in the first BN/2
      // columns of S_g), B = V_j as an MN-major operand, K = 112 keys
      auto issue_pv = [&](int j) {
        const uint32_t vbase = smem_u32(tile_v(j));
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = sdesc(vbase + k * 16 * SW, BN * SW, 8 * SW);
          mma_bf16_ts(t_g + C::O_COL, t_g + k * 8, bd, IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
        }
      };
      // Step k of group g issues PV_g(k-1) (k > 0) and QK_g(k) (k < n_g), once
      // fusion step k has put V_{k-1} and K_k in place.  The two issuers take
      // turns, group 0's step k before group 1's: the turn is one more arrival
      // on the other group's p_full, passed once a step's PV products are
      // issued, so that each group's softmax overlaps the other group's
      // products.  Group 1 of a one-head CTA may read one tile more than
      // group 0: group 0 then passes the turn once more, and that last tile's
      // slots are never refilled, so their empty phases are never awaited.
      const int ng = n_tiles(g);
      auto pass_turn = [&]() { mbar_arrive(&p_full[1 - g]); };
      auto step_operands = [&](int k) {
        return wait(&step_ready[k % NSR], (uint32_t)(k / NSR) & 1u);
      };
      bool ok = wait(q_ready, 0) && step_operands(0);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        mma_commit(&s_full[g]);
        if (g == 1) pass_turn();   // group 0's step 1 follows group 1's step 0
      }
      for (int j = 0; ok && j < ng; ++j) {
        const bool more = j + 1 < ng;
        // every wait comes before the step's first product
        if (!wait(&p_full[g], (uint32_t)j & 1u) || !step_operands(j + 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(j);
        pass_turn();
        if (more) issue_qk(j + 1);
        mma_commit(&s_full[g]);
        // V_j was read by this step's PV products, K_j by the previous step's
        mma_commit(&v_empty[j % NSV]);
        mma_commit(&k_empty[j % NSK]);
      }
      // pass group 1's extra turn once the phase before has completed (an
      // early arrival would count towards that phase)
      if (g == 0)
        for (int j = ng; ok && j < n_tiles(1); ++j) {
          ok = wait(&p_full[1], (uint32_t)(j - 1) & 1u);
          if (ok) pass_turn();
        }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_SOFTMAX));
    // ---------------- softmax warpgroup of group g ----------------
    const int g = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int m_row = g_row0(g) + row;       // query row within the chunk
    const int qpos = p.q_start + m_row;      // its cache position
    const int pos_g = p.q_start + g_row0(g);
    const int ng = n_tiles(g);
    const bool row_valid = m_row < p.S;
    const uint32_t t_s = tmem + ((uint32_t)(quarter * 32) << 16) + g * GROUP_COLS;
    const uint32_t t_o = t_s + C::O_COL;
    {
      // this thread's Q row into tensor memory as D/2 packed bf16 pairs
      // (rows beyond the chunk, and the columns past D/2, are zero)
      const uint4* qrow = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(p.q) + (((size_t)b * H_q + g_head(g)) * p.S + m_row) * D);
      float qw[C::Q_COLS];
#pragma unroll
      for (int i = 0; i < C::Q_COLS / 4; ++i) {
        const uint4 x = (row_valid && i < D / 8) ? qrow[i] : make_uint4(0, 0, 0, 0);
        qw[4 * i] = __uint_as_float(x.x);
        qw[4 * i + 1] = __uint_as_float(x.y);
        qw[4 * i + 2] = __uint_as_float(x.z);
        qw[4 * i + 3] = __uint_as_float(x.w);
      }
#pragma unroll
      for (int c = 0; c < C::Q_COLS; c += 16) tmem_st16(t_s + C::Q_COL + c, qw + c);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < ng; ++j) {
      const int n0 = (j0 + j) * BN;
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, wait(&s_full[g], (uint32_t)j & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c = 0; c + 32 <= BN; c += 32) tmem_ld32(t_s + c, sv + c);
      tmem_ld16(t_s + 96, sv + 96);
      tmem_wait_ld();
      // masking needed: the causal diagonal, the key extent, or (window) the
      // lowest row-window start of the tile (warp-uniform)
      const bool diag = n0 + BN > pos_g || n0 + BN > S_kv || (W > 0 && n0 < pos_g + BM - W);
      if (diag) {
        // visible keys of this row, as tile columns: lo <= c < hi
        const int hi = min(qpos + 1, S_kv) - n0;
        const int lo = W > 0 ? qpos - W + 1 - n0 : INT_MIN;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= hi || c < lo) sv[c] = -INFINITY;
      }
      // row max of the raw scores (the scale is positive, so it commutes):
      // four independent chains
      float mx[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) mx[r] = fmaxf(sv[2 * r], sv[2 * r + 1]);
#pragma unroll
      for (int c = 8; c < BN; c += 8) {
#pragma unroll
        for (int r = 0; r < 4; ++r) mx[r] = fmax3f(mx[r], sv[c + 2 * r], sv[c + 2 * r + 1]);
      }
      const float mt_row = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
      // Keep a stale max until it is exceeded by more than 2^8: P stays
      // below 256 (exact in bf16 and fp32) and O needs no rescaling.
      const float m_new = mt_row > m_run + RESCALE_SLACK ? mt_row : m_run;
      const float alpha = fast_exp2(m_run - m_new);
      const float neg_m = -m_new;
      float ps[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) ps[r] = 0.f;
      // P over the S tile just read: 56 packed columns, stored 16 + 16 + 16 + 8
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        constexpr int W16 = 16;
        const int ncol = qt < 3 ? W16 : 8;
        float pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c >= ncol) break;
          const int cc = qt * 32 + 2 * c;
          // x = s * scale - m for two scores with one packed FMA; exp2(-inf) = 0
          float x0 = neg_m, x1 = neg_m;
          fma2(x0, x1, sv[cc], sv[cc + 1], p.scale_log2, p.scale_log2);
          const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
          const int r = c & 3;
          add2(ps[2 * r], ps[2 * r + 1], e0, e1);
          __nv_bfloat162 v2 = __floats2bfloat162_rn(e0, e1);
          pk[c] = __uint_as_float(*reinterpret_cast<uint32_t*>(&v2));
        }
        if (qt < 3)
          tmem_st16(t_s + qt * 16, pk);
        else
          tmem_st8(t_s + 48, pk);
      }
      const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
        // O_g holds every PV product up to tile j-1 (s_full of tile j); the
        // next one is issued only after p_full below
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          float ov[16];
          tmem_ld16(t_o + c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] *= alpha;
          tmem_st16(t_o + c, ov);
        }
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[g]);
    }
    // the commit after the last PV product is phase ng of s_full[g]
    if (ok && __all_sync(0xffffffffu, wait(&s_full[g], (uint32_t)ng & 1u))) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            (((size_t)b * H_q + g_head(g)) * p.S + m_row) * D;
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

  // (a producer that stopped early has let its copies in flight land)
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out somewhere, so no role may have awaited the last copies
    // and products: each TMA producer lets its copies in flight land (the
    // last tiles of each of its rings; an older tile was consumed before its
    // slot was refilled) and each issuer lets its own products finish,
    // before the CTA frees tensor memory and exits.
    if ((warp == C::K_PRODUCER_WARP || warp == C::V_PRODUCER_WARP) && lane == 0) {
      const bool is_k = warp == C::K_PRODUCER_WARP;
      const int n0s = is_k ? NSK : NSV;
      uint64_t* f0 = is_k ? k_full : v_full;
      uint64_t* f1 = is_k ? k1_full : v1_full;
      const int issued = sm_issued[is_k ? 0 : 1];
      const int t0 = (issued + 1) / 2, t1 = issued / 2;   // tiles issued per ring
      for (int j = max(0, t0 - n0s); j < t0; ++j)
        (void)mbar_wait_bounded(&f0[j % n0s], (uint32_t)(j / n0s) & 1u, kDrainLimitNs);
      for (int j = max(0, t1 - NS1); j < t1; ++j)
        (void)mbar_wait_bounded(&f1[j % NS1], (uint32_t)(j / NS1) & 1u, kDrainLimitNs);
    }
    if (warp >= C::MMA_WARP && warp < C::MMA_WARP + NG && lane == 0) {
      mma_commit(&mma_drain[warp - C::MMA_WARP]);
      (void)mbar_wait_bounded(&mma_drain[warp - C::MMA_WARP], 0, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_fused_wide(const PrefillArgs& a, cudaStream_t stream) {
  using C = FwCfg<D>;
  FwMaps maps;
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
  bool ok = make_map(&maps.k0, a.k[0], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.k1, a.k[1], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.v0, a.v[0], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.v1, a.v[1], D, map_rows, units, kv_plane, BN);
  if (!ok) return cudaErrorInvalidValue;
  FwParams p;
  p.a0 = a.a[0];
  p.a1 = a.a[1];
  p.b0 = a.b[0];
  p.b1 = a.b[1];
  p.q = a.q;
  p.out = a.out;
  p.status = a.status;
  p.wait_limit = a.wait_limit;
  p.H_kv = a.kv_heads;
  p.G = a.group;
  p.S = a.S;
  p.q_start = a.q_start;
  p.S_kv = S_kv;
  p.window = a.window;
  p.ring = a.ring;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  auto kern = prefill_fused_wide_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel must fit the launch allocation, or
  // the softmax warpgroups' increase would never be granted: refuse instead.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if ((long long)fa.numRegs * C::THREADS < C::REGS_SPLIT) return cudaErrorNotSupported;
  // one CTA per (unit, 256 query rows of one head or 128 rows of two heads)
  const int rows_per_cta = a.group == 2 ? BM : NG * BM;
  dim3 grid((unsigned)units, (unsigned)((a.S + rows_per_cta - 1) / rows_per_cta));
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_fused_wide_launch(const PrefillArgs& a, cudaStream_t stream) {
  if (a.nsrc != 2 || (a.group != 1 && a.group != 2)) return cudaErrorNotSupported;
  switch (a.head_dim) {
    case 64: return launch_fused_wide<64>(a, stream);
    case 80: return launch_fused_wide<80>(a, stream);
    case 96: return launch_fused_wide<96>(a, stream);
    default: return cudaErrorNotSupported;   // D = 128: Q does not fit beside S and O
  }
}

}  // namespace fkv
