// Causal prefill attention over ONE key/value source per layer (vanilla
// layers, the Lite upper layers that read K^n / V^1, FusedKV slides Eq.(6),
// and the scaled single-source form) on the tcgen05 tensor cores of sm_103a,
// with 128-key tiles.
//
// What one call computes: for every sequence b, query head h (KV head
// kh = h / G) and query position m of the chunk
//     o_{h,m} = sum_{t <= m, t > m - W} softmax_t(scale * q_{h,m} . K_t) V_t
// (W = infinity unless the layer has a sliding window).
//
// Design.  A CTA owns two "groups" of 128 query rows that read the same keys:
// the two query heads of one KV head (G = 2), or two consecutive 128-row tiles
// of one head (G = 1).  Each group has one softmax warpgroup (a thread per
// query row, i.e. per TMEM lane) and 256 tensor-memory columns: S_g (128 fp32
// columns, overwritten in place by P_g as bf16) and O_g (D columns).
//  * A TMA producer warp loads both groups' Q once and K/V tiles of 128 keys
//    (64-byte swizzle) into a ring of NS stages.
//  * The MMA warp, per key tile j and group g, waits for P_g(j), then issues
//    O_g += P_g V_j (A operand read from tensor memory) and S_g = Q_g K_{j+1}^T,
//    and commits both to s_full[g].  The tensor pipe executes in order, so the
//    QK product that overwrites S_g/P_g runs after the PV product that reads
//    P_g; and when s_full[g] completes, O_g holds every product before tile
//    j+1, so the softmax may rescale it.
//  * The groups alternate on the tensor pipe: while one group's softmax works
//    on its scores, the pipe runs the other group's PV and QK products.
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
constexpr int BN = 128;          // keys per tile
constexpr int NG = 2;            // groups per CTA
constexpr int GROUP_COLS = 256;  // TMEM columns per group: S/P (BN) then O (D)
constexpr int SW = kSW;
constexpr int SWE = kSWE;
constexpr int SMEM_LIMIT = 232448;   // opt-in dynamic shared memory per CTA (227 KB)
constexpr float RESCALE_SLACK = 8.f; // log2 growth of the running max tolerated before O is rescaled

template <int D>
struct WideCfg {
  static constexpr int CB = (D + SWE - 1) / SWE;     // 32-element column blocks
  static constexpr int Q_BYTES = CB * BM * SW;       // one group's Q tile
  static constexpr int KV_BYTES = CB * BN * SW;      // one K or V tile
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int FIXED = NG * Q_BYTES + 2 * D * 4 + 1024;
  static constexpr int NS_FIT = (SMEM_LIMIT - 512 - FIXED) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int SOFTMAX_WARPS = 4 * NG;
  // control warpgroup: the TMA producer, one MMA-issuing warp per group and
  // an idle warp (register reallocation works per warpgroup).  Each group has
  // its own issuing thread: a thread that waits on an mbarrier right after
  // issuing MMAs lets the tensor pipe run dry, and with two issuers the other
  // group's products fill that gap.
  static constexpr int PRODUCER_WARP = SOFTMAX_WARPS;
  static constexpr int MMA_WARP = PRODUCER_WARP + 1;   // + g for group g
  static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 4);
  // registers per thread: 168 at launch (65536 / 384, in steps of 8); the
  // control warpgroup gives up to 40 and the softmax warpgroups take 232:
  // 2 * 128 * 232 + 128 * 40 = 384 * 168, so the increase is always granted
  // (at 224 the softmax spilled a few values; 232 holds them)
#ifdef FKV_PW_REGS_CONTROL
  static constexpr int REGS_CONTROL = FKV_PW_REGS_CONTROL;   // tuning sweeps
  static constexpr int REGS_SOFTMAX = FKV_PW_REGS_SOFTMAX;
#else
  static constexpr int REGS_CONTROL = 40;
  static constexpr int REGS_SOFTMAX = 232;
#endif
  static_assert(NG * 128 * REGS_SOFTMAX + 128 * REGS_CONTROL <= THREADS * 168,
                "register split above the launch allocation");
  static constexpr size_t SMEM = 512 + (size_t)FIXED + (size_t)NS * STAGE;
  static_assert(NS >= 2, "shared memory too small for two K/V stages");
};

struct WideParams {
  const float* a;   // scaled form: S = (Q (.) a) K^T, O = (P V) (.) b; else null
  const float* b;
  void* out;
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

struct WideMaps {
  CUtensorMap q, k, v;
};

template <int D>
__global__ void __launch_bounds__(WideCfg<D>::THREADS, 1)
    prefill_wide_kernel(const __grid_constant__ WideMaps maps, const WideParams p) {
  using C = WideCfg<D>;
  constexpr int CB = C::CB, NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  // 512-byte alignment: the period of the 64-byte swizzle pattern
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 511) &
                                             ~uintptr_t(511));
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + NG * C::Q_BYTES;
  float* sW = reinterpret_cast<float*>(sKV + NS * C::STAGE);   // a then b (scaled form)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW + 2 * D);
  uint64_t* bar_q = bars;
  uint64_t* q_ready = bar_q + 1;
  uint64_t* kv_full = q_ready + 1;
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;   // [NG]
  uint64_t* p_full = s_full + NG;     // [NG]
  uint64_t* mma_drain = p_full + NG;  // [NG] an issuer's last products, after an abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + NG);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* sm_issued = reinterpret_cast<int*>(tmem_slot + 2);   // K/V stages the producer issued

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
  const bool scaled = p.a != nullptr;
  const unsigned long long wlim = wait_limit_ns(p.wait_limit);

  auto stage_k = [&](int s) { return sKV + (size_t)s * C::STAGE; };
  auto stage_v = [&](int s) { return sKV + (size_t)s * C::STAGE + C::KV_BYTES; };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait_bounded(bar, parity, wlim)) return true;
    *abort_flag = 1;
    flag_status(p.status, kDevTimeout);
    return false;
  };

  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(q_ready, 128 * NG);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], NG);   // one commit per group that reads the tile
    }
    for (int g = 0; g < NG; ++g) {
      mbar_init(&s_full[g], 1);
      // the group's 128 softmax threads, plus the other group's issuer once
      // its previous step's PV products are queued (the turn)
      mbar_init(&p_full[g], 129);
      mbar_init(&mma_drain[g], 1);
    }
    *abort_flag = 0;
    *sm_issued = 0;
    fence_mbar_init();
  }
  if (scaled) {
    for (int i = tid; i < D; i += C::THREADS) {
      sW[i] = p.a[kh * D + i];
      sW[D + i] = p.b[kh * D + i];
    }
  }
  if (warp == C::MMA_WARP) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::SOFTMAX_WARPS) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CONTROL));
    if (warp == C::PRODUCER_WARP) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, NG * C::Q_BYTES);
      for (int g = 0; g < NG; ++g)
        for (int cb = 0; cb < CB; ++cb)
          tma_load_3d(sQ + g * C::Q_BYTES + cb * BM * SW, &maps.q, cb * SWE, g_row0(g),
                      b * H_q + g_head(g), bar_q);
      int issued = 0;
      for (int j = 0; j < n_max; ++j) {
        const int s = j % NS, u = j / NS;
        if (u > 0 && !wait(&kv_empty[s], (uint32_t)(u - 1) & 1u)) break;
        const int n0 = (j0 + j) * BN;
        // the tile's first cache row: in a ring, whole tiles never wrap
        const int ky = p.ring > 0 ? n0 % p.ring : n0;
        mbar_arrive_expect_tx(&kv_full[s], C::STAGE);
        for (int cb = 0; cb < CB; ++cb) {
          tma_load_3d(stage_k(s) + cb * BN * SW, &maps.k, cb * SWE, ky, unit, &kv_full[s]);
          tma_load_3d(stage_v(s) + cb * BN * SW, &maps.v, cb * SWE, ky, unit, &kv_full[s]);
        }
        issued = j + 1;
      }
      *sm_issued = issued;
    }
  } else if (warp < C::MMA_WARP + NG) {
    // ---------------- MMA issuer of group g ----------------
    const int g = warp - C::MMA_WARP;
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, true);
      const uint32_t t_g = tmem + g * GROUP_COLS;
      const uint32_t qbase = smem_u32(sQ + g * C::Q_BYTES);
      // S_g = Q_g K_j^T: M = 128 rows, N = 128 keys, K = D in steps of 16
      auto issue_qk = [&](int j) {
        const uint32_t kbase = smem_u32(stage_k(j % NS));
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (uint32_t)(k & 1) * 32;
          const uint64_t ad = sdesc(qbase + (k >> 1) * BM * SW + off, 16, 8 * SW);
          const uint64_t bd = sdesc(kbase + (k >> 1) * BN * SW + off, 16, 8 * SW);
          mma_bf16(t_g, ad, bd, IDESC_QK, k > 0);
        }
      };
      // O_g += P_g V_j: A = P_g (bf16, two per column, in the first BN/2
      // columns of S_g), B = V_j as an MN-major operand, K = 128 keys
      auto issue_pv = [&](int j) {
        const uint32_t vbase = smem_u32(stage_v(j % NS));
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = sdesc(vbase + k * 16 * SW, BN * SW, 8 * SW);
          mma_bf16_ts(t_g + BN, t_g + k * 8, bd, IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
        }
      };
      // Step k of group g issues PV_g(k-1) (k > 0) and QK_g(k) (k < n_g).
      // The two issuers take turns, group 0's step k before group 1's (the
      // turn passes once a step's PV products are issued), so that the tensor
      // pipe alternates between the groups and each group's softmax overlaps
      // the other group's products (without the ordering the groups fall
      // into step and their softmaxes run side by side).  The turn is one
      // more arrival on the other group's p_full: phase j of p_full[g]
      // completes when P_g(j) is in place and the other issuer has queued
      // its step before (group 1's step j+1 follows group 0's, group 0's
      // step j+1 follows group 1's step j), so one wait covers both.
      // Group 1 of a one-head CTA may read one tile more than group 0 (its
      // rows end 128 positions later): group 0 then passes the turn once
      // more, and that last tile's slot is never refilled, so its kv_empty
      // phase is never awaited.
      const int ng = n_tiles(g);
      auto pass_turn = [&]() { mbar_arrive(&p_full[1 - g]); };
      bool ok = wait(scaled ? q_ready : bar_q, 0) && wait(&kv_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        mma_commit(&s_full[g]);
        if (g == 1) pass_turn();   // group 0's step 1 follows group 1's step 0
      }
      for (int j = 0; ok && j < ng; ++j) {
        const bool more = j + 1 < ng;
        if (!wait(&p_full[g], (uint32_t)j & 1u) ||
            (more && !wait(&kv_full[(j + 1) % NS], (uint32_t)((j + 1) / NS) & 1u))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(j);
        pass_turn();
        if (more) issue_qk(j + 1);
        mma_commit(&s_full[g]);
        mma_commit(&kv_empty[j % NS]);
      }
      // group 1 of a one-head CTA may take one step more than group 0: pass
      // its turn too, once the phase before has completed (an early arrival
      // would count towards that phase)
      if (g == 0)
        for (int j = ng; ok && j < n_tiles(1); ++j) {
          ok = wait(&p_full[1], (uint32_t)(j - 1) & 1u);
          if (ok) pass_turn();
        }
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
    const uint32_t t_s = tmem + ((uint32_t)(quarter * 32) << 16) + g * GROUP_COLS;
    const uint32_t t_o = t_s + BN;
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    if (scaled) {
      // this thread's Q row times a, in place (swizzled 16-byte chunks)
      ok = wait(bar_q, 0);
      uint8_t* qg = sQ + g * C::Q_BYTES;
      for (int cb = 0; ok && cb < CB; ++cb) {
        for (int lc = 0; lc < 4; ++lc) {
          const int col = cb * SWE + lc * 8;
          if (col >= D) continue;
          uint4* pq = reinterpret_cast<uint4*>(qg + cb * BM * SW + swz64(row, lc));
          float f[8];
          unpack16<__nv_bfloat16>(*pq, f);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 v2 = __floats2bfloat162_rn(f[2 * e] * sW[col + 2 * e],
                                                      f[2 * e + 1] * sW[col + 2 * e + 1]);
            o[e] = *reinterpret_cast<uint32_t*>(&v2);
          }
          *pq = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
      ok = __all_sync(0xffffffffu, ok);
    }
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
      for (int c = 0; c < BN; c += 32) tmem_ld32(t_s + c, sv + c);
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
      // eight independent chains over column pairs
      float mx[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) mx[r] = fmaxf(sv[2 * r], sv[2 * r + 1]);
#pragma unroll
      for (int c = 16; c < BN; c += 16) {
#pragma unroll
        for (int r = 0; r < 8; ++r) mx[r] = fmax3f(mx[r], sv[c + 2 * r], sv[c + 2 * r + 1]);
      }
      const float mt_row = fmaxf(fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]), mx[6]),
                                 mx[7]) * p.scale_log2;
      // Keep a stale max until it is exceeded by more than 2^8: P stays
      // below 256 (exact in bf16 and fp32) and O needs no rescaling.
      const float m_new = mt_row > m_run + RESCALE_SLACK ? mt_row : m_run;
      const float alpha = fast_exp2(m_run - m_new);
      const float neg_m = -m_new;
      // row sum in four independent packed accumulators
      float ps[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) ps[r] = 0.f;
      // P over the S tile just read, in quarters of 32 keys (16 columns)
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        float pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int cc = qt * 32 + c;
          // x = s * scale - m for two scores with one packed FMA; exp2(-inf) = 0
          float x0 = neg_m, x1 = neg_m;
          fma2(x0, x1, sv[cc], sv[cc + 1], p.scale_log2, p.scale_log2);
          const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
          const int r = (c >> 1) & 3;
          add2(ps[2 * r], ps[2 * r + 1], e0, e1);
          __nv_bfloat162 v2 = __floats2bfloat162_rn(e0, e1);
          pk[c / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&v2));
        }
        tmem_st16(t_s + qt * 16, pk);
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
      const bool row_valid = m_row < p.S;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float ov[16];
        tmem_ld16(t_o + c, ov);
        tmem_wait_ld();
        if (scaled) {
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] *= sW[D + c + e];
        }
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
    // last NS stages; every older stage was consumed before its slot was
    // refilled) and each issuer lets its own products finish, before the CTA
    // frees tensor memory and exits.
    if (warp == C::PRODUCER_WARP && lane == 0) {
      (void)mbar_wait_bounded(bar_q, 0, kDrainLimitNs);
      const int issued = *sm_issued;
      for (int j = max(0, issued - NS); j < issued; ++j)
        (void)mbar_wait_bounded(&kv_full[j % NS], (uint32_t)(j / NS) & 1u, kDrainLimitNs);
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
cudaError_t launch_wide(const PrefillArgs& a, cudaStream_t stream) {
  using C = WideCfg<D>;
  WideMaps maps;
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
  bool ok = make_map(&maps.q, a.q, D, a.S, (long long)a.batch * a.kv_heads * a.group,
                     (size_t)a.S * D * 2, BM);
  ok = ok && make_map(&maps.k, a.k[0], D, map_rows, units, kv_plane, BN);
  ok = ok && make_map(&maps.v, a.v[0], D, map_rows, units, kv_plane, BN);
  if (!ok) return cudaErrorInvalidValue;
  WideParams p;
  p.a = a.a[0];
  p.b = a.b[0];
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
  auto kern = prefill_wide_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel must fit the launch allocation, or
  // the softmax warpgroups' increase would never be granted: refuse instead.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if ((long long)fa.numRegs * C::THREADS <
      (long long)NG * 128 * C::REGS_SOFTMAX + 128LL * C::REGS_CONTROL)
    return cudaErrorNotSupported;
  // one CTA per (unit, 256 query rows of one head or 128 rows of two heads)
  const int rows_per_cta = a.group == 2 ? BM : NG * BM;
  dim3 grid((unsigned)units, (unsigned)((a.S + rows_per_cta - 1) / rows_per_cta));
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_wide_launch(const PrefillArgs& a, cudaStream_t stream) {
  if (a.nsrc != 1 || (a.group != 1 && a.group != 2)) return cudaErrorNotSupported;
  switch (a.head_dim) {
    case 64: return launch_wide<64>(a, stream);
    case 80: return launch_wide<80>(a, stream);
    case 96: return launch_wide<96>(a, stream);
    case 128: return launch_wide<128>(a, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fkv
