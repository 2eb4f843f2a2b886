// Persistent backward for short sequences: one CTA per SM takes (batch, key/value head,
// 128-key block) units from a device-wide counter until none is left.
//
// Method: the key-block backward of fa_bwd.cu (the textbook gradient with P recomputed
// from the saved log-sum-exp, "FlashAttention-2: atención eficiente en GPU para contextos
// largos", section "Bloques pequeños, normalización global"), with the work split over the
// sequence as well as batch and heads so the GPU stays full (same page, section "Tres
// mejoras en la utilización de la GPU", second point).  With few query steps per key
// block, a CTA that owns one block spends about a third of its time starting (barriers,
// TMEM, K and V from memory, V into TMEM) and finishing (dK and dV out of TMEM and
// stored).  Here a CTA lives for many units and overlaps those phases with its
// neighbours' steps:
//  * warp 12 takes the next unit (one atomic add on the launch's counter), passes it to
//    the other roles through a two-entry queue in shared memory, and loads its K into
//    one of two K buffers and its V into a V buffer of its own while the current unit's
//    steps run; the Q / dO / lse / D ring runs on across units;
//  * warp 13 issues the next unit's first S^T = K Q^T before the current unit's last
//    gradient products, and its first dP^T once V is in TMEM, so the tensor pipe goes
//    from one unit to the next without draining;
//  * warpgroup 1 copies V into TMEM as soon as the previous unit's last dP^T has been
//    read; warpgroup 2 (the dQ^T reader) reads dK and dV out of TMEM after each unit's
//    last gradient products, frees the accumulators for the next unit's first ones, and
//    stores dK through the finished unit's K buffer and dV through the V buffer (whose
//    next unit's V is by then in TMEM), each warp its 32 key rows by TMA stores, before
//    both buffers go back to the producer.
// Units are taken in the order of the one-CTA-per-block grid (with the causal mask the
// heaviest first), so the dynamic counter balances the tail.  The counter pair {next,
// done} is picked per launch from the ring the persistent forward uses; the last CTA to
// finish puts it back to {0, 0}.
#include "fa_internal.h"
#include "fa_bwd_common.cuh"
#include "sm100_ptx.cuh"

namespace fa {

template <int D>
struct BpCfg {
  static constexpr int CHUNKS = D / 64;           // 128-byte swizzle column chunks
  static constexpr int KV_TILE = 128 * D * 2;     // K or V tile
  static constexpr int KV_CHUNK = 128 * 128;      // 128 rows x 128 B
  static constexpr int Q_CHUNK = 64 * 128;        // 64 rows x 128 B
  static constexpr int Q_TILE = 64 * D * 2;       // Q or dO tile
  static constexpr int DS_TILE = 128 * 64 * 2;    // dS^T tile, 128 keys x 64 queries, 16-bit
  static constexpr int STG = (D == 128) ? 3 : 6;  // Q/dO/lse/D stages
  static constexpr int THREADS = 512;
  // control warps 80, softmax warpgroups 160, dQ warpgroup 112 registers
  static constexpr int REG_SPLIT = 128 * 80 + 256 * 160 + 128 * 112;
  static_assert(REG_SPLIT <= THREADS * 128, "register split above the launch allocation");
  static constexpr bool DQ_TMA = (D == 64);       // d=64: dQ^T added by TMA tensor reductions
  static constexpr bool DP_FIRST = (D == 128);    // issue order within a unit, as in fa_bwd.cu
  static constexpr int DQ_HALF = D * 128;
  static constexpr int EPC = (D == 128) ? 64 : 32;  // dK / dV columns per TMEM read in the epilogue
  // barriers: sdp_full, dp_free, ds_ready[2], ds_free[2], dq_full[2], dq_free, final,
  // k_full[2], k_empty[2], v_full, v_empty, v_tmem, acc_done, acc_free, uq_full[2],
  // uq_empty[2], then the stage ring's full[STG] / empty[STG]
  static constexpr int B_SDP = 0, B_DPFREE = 1, B_DSREADY = 2, B_DSFREE = 4, B_DQFULL = 6, B_DQFREE = 8,
                       B_FINAL = 9, B_KFULL = 10, B_KEMPTY = 12, B_VFULL = 14, B_VEMPTY = 15, B_VTM = 16,
                       B_ACC = 17, B_ACCFREE = 18, B_UF = 19, B_UE = 21, B_STFULL = 23;
  static constexpr int NBARS = 23 + 2 * STG;
  // shared memory (offsets from the 1024-aligned base): K[2], V, Q[STG], dO[STG], dS^T[2],
  // the d=64 dQ^T staging, [STG][2][64] floats (-lse*log2e, -D), barriers, a few words
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = 2 * KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STG * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + STG * Q_TILE;
  static constexpr int OFF_DQS = OFF_DS + 2 * DS_TILE;
  static constexpr int DQS_BYTES = DQ_TMA ? 2 * DQ_HALF : 0;
  static constexpr int OFF_LD = OFF_DQS + DQS_BYTES;
  static constexpr int OFF_BAR = OFF_LD + STG * 2 * 64 * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + 8 * NBARS + 64;  // 1024: alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  // tensor memory as in fa_bwd.cu: S^T[2] (P^T | dS^T, then dQ^T), dP^T, V, dV, dK
  static constexpr uint32_t T_S = 0, T_DP = 128, T_V = 192, T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
};

// One unit: keys [128 jb, 128 jb + 128) of (b, hkv), walked against every query head of
// the GQA group and every 64-query block that sees them (T steps).
struct BpUnit {
  int b, hkv, k0, qb0, nq, T;
};

template <bool CAUSAL>
__device__ __forceinline__ BpUnit bp_decode(int u, const BwdParams& p, int G) {
  // the one-CTA-per-block grid's order: key blocks of a (batch, key/value head) pair
  // consecutive; with the mask, at least 32 key blocks and at most 64 pairs, block jb of
  // every pair before block jb + 1 of any
  const int nkb = (p.N + 127) / 128;
  const int BHK = p.B * p.Hkv;
  const bool kb_major = CAUSAL && nkb >= 32 && BHK <= 64;
  const int jb = kb_major ? u / BHK : u % nkb;
  const int bhk = kb_major ? u % BHK : u / nkb;
  BpUnit w;
  w.hkv = bhk % p.Hkv;
  w.b = bhk / p.Hkv;
  w.k0 = 128 * jb;
  w.qb0 = CAUSAL ? 2 * jb : 0;  // the first 64-query block that sees key k0
  w.nq = (p.N + 63) / 64 - w.qb0;
  w.T = G * w.nq;
  return w;
}

// Row r of a D-column fp32 accumulator in TMEM (from column address `col`, lane r), times
// `mul` if SCALED, rounded to 16 bits into row r of a staging tile laid out as the K / V
// loads (64-column chunks of 128 rows x 128 B, 128-byte swizzle).
template <int D, bool BF16, bool SCALED>
__device__ __forceinline__ void bp_stage_rows(uint32_t col, float mul, uint8_t* stage, int r) {
  constexpr int EPC = BpCfg<D>::EPC;
  const uint64_t mul2 = f2pack(mul, mul);
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += EPC) {
    uint32_t v[EPC];
#pragma unroll
    for (int h = 0; h < EPC / 32; ++h) tmem_ld32(col + c0 + 32u * h, v + 32 * h);
    tmem_wait_ld();
    uint8_t* rowp = stage + (c0 / 64) * BpCfg<D>::KV_CHUNK + r * 128;
#pragma unroll
    for (int u8 = 0; u8 < EPC / 8; ++u8) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a = __uint_as_float(v[8 * u8 + 2 * i]), b = __uint_as_float(v[8 * u8 + 2 * i + 1]);
        if (SCALED) f2unpack(fmul2(f2pack(a, b), mul2), a, b);
        pk[i] = pack_half2<BF16>(a, b);
      }
      const int unit = (c0 % 64) / 8 + u8;
      *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

template <int D, bool BF16, bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(512, 1) fa_bwd_persistent(const __grid_constant__ BwdParams p, unsigned* sched,
                                                            int units) {
  using C = BpCfg<D>;
  extern __shared__ uint8_t smem_raw_bp[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_bp) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* dq_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);  // d=64 dQ warps gave up
  volatile int* uq = reinterpret_cast<volatile int*>(tmem_slot + 3);       // [2] unit queue
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * i; };
  const uint32_t sdp_full = bar(C::B_SDP), dp_free = bar(C::B_DPFREE), dq_free = bar(C::B_DQFREE);
  const uint32_t final_bar = bar(C::B_FINAL), v_full = bar(C::B_VFULL), v_empty = bar(C::B_VEMPTY);
  const uint32_t v_tmem = bar(C::B_VTM), acc_done = bar(C::B_ACC), acc_free = bar(C::B_ACCFREE);
  auto ds_ready = [&](int b) { return bar(C::B_DSREADY + b); };
  auto ds_free = [&](int b) { return bar(C::B_DSFREE + b); };
  auto dq_full = [&](int b) { return bar(C::B_DQFULL + b); };
  auto k_full = [&](int b) { return bar(C::B_KFULL + b); };
  auto k_empty = [&](int b) { return bar(C::B_KEMPTY + b); };
  auto uq_full = [&](int b) { return bar(C::B_UF + b); };
  auto uq_empty = [&](int b) { return bar(C::B_UE + b); };
  auto st_full = [&](int s) { return bar(C::B_STFULL + s); };
  auto st_empty = [&](int s) { return bar(C::B_STFULL + C::STG + s); };
  constexpr unsigned FULL = 0xffffffffu;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *dq_fail = 0;
    mbar_init(sdp_full, 1);
    mbar_init(dp_free, 256);
    mbar_init(dq_free, 128);
    mbar_init(final_bar, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 128 + 4);  // wg1's copy into TMEM and the 4 epilogue warps' staging
    mbar_init(v_tmem, 128);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(ds_ready(i), 256);
      mbar_init(ds_free(i), 1);
      mbar_init(dq_full(i), 1);
      mbar_init(k_full(i), 1);
      mbar_init(k_empty(i), 1 + 4);  // the MMA's release and the 4 epilogue warps' (staging)
      mbar_init(uq_full(i), 1);
      mbar_init(uq_empty(i), 13);  // the MMA warp's leader and lane 0 of the 12 other consumer warps
    }
    for (int s = 0; s < C::STG; ++s) {
      mbar_init(st_full(s), 1);
      mbar_init(st_empty(s), 1);
    }
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;
  const volatile int* no_abort = nullptr;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.err, kDevErrTimeout);
  };
  const int wg = warp >> 2;                        // 0,1: softmax; 2: dQ and dK / dV out; 3: control
  const int r = (warp & 3) * 32 + lane;            // TMEM lane: key row (wg 0,1,2 epilogue) or d index (wg 2 dQ^T)
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
  // queue entry `n` (warp-uniform); lane 0 (or the given lane) releases it for the warp
  auto pop = [&](int n, int& u, bool release) {
    const int slot = n & 1;
    if (!__all_sync(FULL, mbar_wait(uq_full(slot), (n >> 1) & 1, abort_flag, lim))) return false;
    u = uq[slot];
    __syncwarp();
    if (release) mbar_arrive(uq_empty(slot));
    return true;
  };

  if (wg == 3) {
    setmaxnreg_dec<80>();
    const bool leader = elect_one();
    if (warp == 12) {
      // ------------------------------------------------- scheduler + TMA producer
      const int lead_lane = __ffs(__ballot_sync(FULL, leader)) - 1;
      if (leader) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_do);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        if (C::DQ_TMA && DQ) tma_prefetch_desc(&p.tm_dq);
      }
      bool ok = true;
      int ul = 0;  // queue entries pushed
      int kiss = 0, viss = 0, g = 0;  // K, V and step loads issued
      for (;;) {
        int u = 0;
        if (leader) u = static_cast<int>(atomicAdd(sched, 1u));
        u = __shfl_sync(FULL, u, lead_lane);
        if (u >= units) u = -1;
        const int slot = ul & 1;
        if (ul >= 2 && !__all_sync(FULL, mbar_wait(uq_empty(slot), ((ul >> 1) - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (leader) {
          uq[slot] = u;
          mbar_arrive(uq_full(slot));
        }
        ++ul;
        if (u < 0) break;
        const BpUnit w = bp_decode<CAUSAL>(u, p, G);
        // K into buffer kiss & 1, free once the MMAs of the unit before last are done
        const int kb = kiss & 1;
        if (kiss >= 2 && !__all_sync(FULL, mbar_wait(k_empty(kb), ((kiss >> 1) - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(k_full(kb), C::KV_TILE);
          for (int ch = 0; ch < C::CHUNKS; ++ch)
            tma_load_4d(sbase + C::OFF_K + kb * C::KV_TILE + ch * C::KV_CHUNK, &p.tm_k, k_full(kb), ch * 64, w.hkv,
                        w.k0, w.b);
        }
        ++kiss;
        // V, free once the previous unit's V has been copied into TMEM
        if (viss >= 1 && !__all_sync(FULL, mbar_wait(v_empty, (viss - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(v_full, C::KV_TILE);
          for (int ch = 0; ch < C::CHUNKS; ++ch)
            tma_load_4d(sbase + C::OFF_V + ch * C::KV_CHUNK, &p.tm_v, v_full, ch * 64, w.hkv, w.k0, w.b);
        }
        ++viss;
        for (int it = 0; it < w.T; ++it) {
          const int s = g % C::STG;
          if (g >= C::STG &&
              !__all_sync(FULL, mbar_wait(st_empty(s), ((g / C::STG) - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          const int hq = w.hkv * G + it / w.nq;
          const int q0 = 64 * (w.qb0 + it % w.nq);
          if (leader) {
            mbar_arrive_expect_tx(st_full(s), 2 * C::Q_TILE + 2 * 256);
            for (int ch = 0; ch < C::CHUNKS; ++ch) {
              tma_load_4d(sbase + C::OFF_Q + s * C::Q_TILE + ch * C::Q_CHUNK, &p.tm_q, st_full(s), ch * 64, hq, q0,
                          w.b);
              tma_load_4d(sbase + C::OFF_DO + s * C::Q_TILE + ch * C::Q_CHUNK, &p.tm_do, st_full(s), ch * 64, hq,
                          q0, w.b);
            }
            const long long row = (static_cast<long long>(w.b) * p.Hq + hq) * p.Npad + q0;
            bulk_load(sbase + C::OFF_LD + s * 512, p.l2vec + row, 256, st_full(s));
            bulk_load(sbase + C::OFF_LD + s * 512 + 256, p.dvec + row, 256, st_full(s));
          }
          ++g;
        }
        if (!ok) break;
      }
      if (!ok) {
        if (leader) fail();
        // let the copies in flight land before the CTA's shared memory goes away
        for (int i = (g > C::STG ? g - C::STG : 0); i < g; ++i)
          mbar_wait(st_full(i % C::STG), (i / C::STG) & 1, no_abort, lim);
        for (int i = (kiss > 2 ? kiss - 2 : 0); i < kiss; ++i) mbar_wait(k_full(i & 1), (i >> 1) & 1, no_abort, lim);
        if (viss > 0) mbar_wait(v_full, (viss - 1) & 1, no_abort, lim);
      }
      // this CTA takes no further unit: the last one to get here resets the counter pair
      if (leader) {
        __threadfence();
        if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
          atomicExch(sched, 0u);
          atomicExch(sched + 1, 0u);
        }
      }
      __syncwarp();
    } else if (warp == 13) {
      // --------------------------------------------------------------- MMA issuer
      constexpr uint32_t bf = BF16 ? 1u : 0u;
      constexpr uint32_t id_sdp = idesc_f16(128, 64, bf, 0, 0);  // S^T, dP^T: M=keys, N=queries
      constexpr uint32_t id_grad = idesc_f16(128, D, bf, 0, 1);  // dV, dK: M=keys, N=d, B MN-major
      constexpr uint32_t id_dq = idesc_f16(128, 64, bf, 1, 1);   // dQ^T: M=d (padded to 128), N=queries
      // descriptor templates; per step only the start-address field (16-byte units) moves
      const uint64_t dK_km = smem_desc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dQ_km = smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dDO_km = smem_desc_sw128(sbase + C::OFF_DO, 16, 1024);
      const uint64_t dQ_mn = smem_desc_sw128(sbase + C::OFF_Q, C::Q_CHUNK, 1024);
      const uint64_t dDO_mn = smem_desc_sw128(sbase + C::OFF_DO, C::Q_CHUNK, 1024);
      const uint64_t dDS_mn = smem_desc_sw128(sbase + C::OFF_DS, 1024, 1024);
      const uint64_t dK_mn = smem_desc_sw128(sbase + C::OFF_K, C::KV_CHUNK, 1024);
      auto u16 = [](int bytes) { return static_cast<uint64_t>(bytes >> 4); };
      // the step whose gradient products are still to be issued
      struct Pending {
        int g, i, un;  // global step, step within its unit, the unit's index in this CTA
        bool last;     // the unit's last step
      };
      // dV += P^T dO, dK += dS^T Q, dQ^T = K^T dS^T of step q; a unit's first gradient
      // products overwrite the accumulators, which the previous unit's epilogue must have
      // read out; its last ones announce dK / dV and release the unit's K buffer
      auto grads = [&](const Pending& q) {
        const int s = q.g % C::STG, bb = q.g & 1, kb = q.un & 1;
        if (!__all_sync(FULL, mbar_wait(ds_ready(bb), (q.g >> 1) & 1, abort_flag, lim))) return false;
        if (q.i == 0 && q.un > 0 && !__all_sync(FULL, mbar_wait(acc_free, (q.un - 1) & 1, abort_flag, lim)))
          return false;
        tc_fence_after();
        if (leader) {
          const uint64_t qs = u16(s * C::Q_TILE);
          // k-step kk covers queries [16 kk, 16 kk + 16): in the S^T buffer, queries
          // [32 h, 32 h + 32) hold P^T in columns [32 h, 32 h + 16) and dS^T in
          // [32 h + 16, 32 h + 32), as 16-bit pairs
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tbase + C::T_DV, tbase + C::T_S + 64u * bb + 32u * (kk / 2) + 8u * (kk % 2),
                   dDO_mn + qs + u16(kk * 2048), id_grad, (q.i > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tbase + C::T_DK, tbase + C::T_S + 64u * bb + 32u * (kk / 2) + 16u + 8u * (kk % 2),
                   dQ_mn + qs + u16(kk * 2048), id_grad, (q.i > 0 || kk > 0));
          mma_commit(st_empty(s));
          // the unit's dK and dV are final once these complete: announce them before the
          // dQ^T product, so that their read-out overlaps it
          if (q.last) mma_commit(acc_done);
          if (DQ) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tbase + C::T_S + 64u * bb, dK_mn + u16(kb * C::KV_TILE + kk * 2048),
                     dDS_mn + u16(bb * C::DS_TILE + kk * 2048), id_dq, kk > 0);
            mma_commit(dq_full(bb));
          }
          mma_commit(ds_free(bb));
          if (q.last) mma_commit(k_empty(kb));  // the unit's last product that reads its K buffer
        }
        return true;
      };
      bool ok = true;
      int ul = 0, un = 0, it = 0, g = 0;
      int u = -1;
      BpUnit w{};
      Pending pend{};
      bool have_pend = false;
      ok = pop(ul++, u, leader);
      if (ok && u >= 0) w = bp_decode<CAUSAL>(u, p, G);
      while (ok) {
        if (u >= 0) {
          const int s = g % C::STG, bb = g & 1, kb = un & 1;
          if (it == 0 && !__all_sync(FULL, mbar_wait(k_full(kb), (un >> 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (!__all_sync(FULL, mbar_wait(st_full(s), (g / C::STG) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          const uint64_t qs = u16(s * C::Q_TILE);
          // S^T(g) overwrites the buffer that held dQ^T(g-2), which must have been read out
          auto issue_s = [&]() {
            if (DQ && g >= 2 && !__all_sync(FULL, mbar_wait(dq_free, (g - 2) & 1, abort_flag, lim))) return false;
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tbase + C::T_S + 64u * bb,
                       dK_km + u16(kb * C::KV_TILE + (kk / 4) * C::KV_CHUNK + (kk % 4) * 32),
                       dQ_km + qs + u16((kk / 4) * C::Q_CHUNK + (kk % 4) * 32), id_sdp, kk > 0);
            }
            return true;
          };
          // dP^T(g) overwrites the columns the previous step's softmax has loaded; a unit's
          // first dP^T waits for its V in TMEM
          auto issue_dp = [&]() {
            if (g > 0 && !__all_sync(FULL, mbar_wait(dp_free, (g - 1) & 1, abort_flag, lim))) return false;
            if (it == 0 && !__all_sync(FULL, mbar_wait(v_tmem, un & 1, abort_flag, lim))) return false;
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ts(tbase + C::T_DP, tbase + C::T_V + 8u * kk,
                       dDO_km + qs + u16((kk / 4) * C::Q_CHUNK + (kk % 4) * 32), id_sdp, kk > 0);
            }
            return true;
          };
          bool issued;
          if (it == 0 && have_pend) {
            // a unit's first step: S^T needs only the unit's K (loaded ahead), so it goes in
            // before the previous unit's last gradient products; dP^T waits for V in TMEM,
            // which follows the previous unit's last softmax step, so it goes in after them
            issued = issue_s() && grads(pend) && issue_dp();
            have_pend = false;
          } else {
            issued = C::DP_FIRST ? (issue_dp() && issue_s()) : (issue_s() && issue_dp());
          }
          if (!issued) {
            ok = false;
            break;
          }
          if (leader) mma_commit(sdp_full);  // covers both products
        }
        if (have_pend && !grads(pend)) {
          ok = false;
          break;
        }
        have_pend = false;
        if (u < 0) break;
        pend.g = g;
        pend.i = it;
        pend.un = un;
        pend.last = it == w.T - 1;
        have_pend = true;
        ++g;
        if (++it == w.T) {
          it = 0;
          ++un;
          if (!pop(ul++, u, leader)) {
            ok = false;
            break;
          }
          if (u >= 0) w = bp_decode<CAUSAL>(u, p, G);
        }
      }
      if (!ok && leader) fail();
      if (leader) mma_commit(final_bar);
      mbar_wait(final_bar, 0, no_abort, lim);
      // The last commits to st_empty, ds_free and k_empty have no consumer; let their
      // arrivals land before the CTA's shared memory (and the barriers in it) goes away.
      if (ok) {
        for (int i = (g > C::STG ? g - C::STG : 0); i < g; ++i)
          mbar_wait(st_empty(i % C::STG), (i / C::STG) & 1, no_abort, lim);
        for (int i = (g > 2 ? g - 2 : 0); i < g; ++i) mbar_wait(ds_free(i & 1), (i >> 1) & 1, no_abort, lim);
        for (int i = (un > 2 ? un - 2 : 0); i < un; ++i) mbar_wait(k_empty(i & 1), (i >> 1) & 1, no_abort, lim);
      }
      __syncwarp();
    }
  } else if (wg < 2) {
    setmaxnreg_inc<160>();
    // ------------------------------------------------------ P^T and dS^T
    // warpgroup wg takes query columns [32 wg, 32 wg + 32) of each 64-column step
    bool ok = true;
    const uint64_t cl2x2 = f2pack(p.scale_log2, p.scale_log2);
    const int cbase = 32 * wg;
    int g = 0;
    for (int n = 0;; ++n) {
      int u = -1;
      if (!pop(n, u, lane == 0)) {
        ok = false;
        break;
      }
      if (u < 0) break;
      const BpUnit w = bp_decode<CAUSAL>(u, p, G);
      const int key = w.k0 + r;
      if (wg == 1) {
        // V row r -> TMEM lane r.  The previous unit's last dP^T, the last product to read
        // V's columns, completed before this warpgroup's last softmax step of that unit.
        if (!__all_sync(FULL, mbar_wait(v_full, n & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        bwd_v_to_tmem<C::CHUNKS>(smem + C::OFF_V, r, tbase + lane_off + C::T_V);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(v_tmem);
        mbar_arrive(v_empty);
      }
      for (int it = 0; it < w.T; ++it, ++g) {
        const int s = g % C::STG, bb = g & 1;
        const int q0 = 64 * (w.qb0 + it % w.nq);
        if (!__all_sync(FULL, mbar_wait(st_full(s), (g / C::STG) & 1, abort_flag, lim) &&
                                  mbar_wait(sdp_full, g & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[32], dpv[32];
        tmem_ld32(tbase + lane_off + C::T_S + 64u * bb + cbase, sv);
        tmem_ld32(tbase + lane_off + C::T_DP + cbase, dpv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(dp_free);
        const float4* nl4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512) + cbase / 4;
        const float4* nd4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512 + 256) + cbase / 4;
        // with the causal mask query column c sees this key iff c >= key - q0
        const int cmin = CAUSAL ? key - q0 - cbase : -(1 << 20);
        // the dS^T buffer of this parity must have been consumed by the MMAs of step g-2
        if (g >= 2 && !__all_sync(FULL, mbar_wait(ds_free(bb), ((g >> 1) - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        uint8_t* rowp = smem + C::OFF_DS + bb * C::DS_TILE + r * 128;
        uint32_t pk[16], dsk[16];
        bwd_p_ds<BF16, CAUSAL, DQ>(sv, dpv, nl4, nd4, cmin, cl2x2, rowp, wg, r, pk, dsk);
        tmem_st16(tbase + lane_off + C::T_S + 64u * bb + cbase, pk);
        tmem_st16(tbase + lane_off + C::T_S + 64u * bb + cbase + 16u, dsk);
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(ds_ready(bb));
      }
      if (!ok) break;
    }
    if (!ok) fail();
  } else {
    setmaxnreg_dec<112>();
    // ----------------------------- dQ^T -> fp32 accumulator; dK, dV out of TMEM
    // dQ^T as in fa_bwd.cu (d=128: thread r = row d of dQ^T, one reduction per query and
    // warp; d=64: staged, TMA tensor reductions).  With d=64 the four warps meet at a
    // named barrier per step, so every exit from the loop is taken by all four together:
    // a warp that gives up records it in dq_fail and still arrives.
    bool ok = true;
    int g = 0;
    // dV of unit n is staged in the V buffer, which V(n + 2) may overwrite only after the
    // stores have read it: the V buffer's release (v_empty) counts these 4 warps besides
    // the copy of V into TMEM, and nothing was staged before the first unit
    if (lane == 0) mbar_arrive(v_empty);
    int u = -1;
    bool got_u = pop(0, u, lane == 0);
    for (int n = 0;; ++n) {
      if (C::DQ_TMA && DQ) {
        if (!got_u && lane == 0) *dq_fail = 1;
        named_bar_sync_n(1, 128);
        if (*dq_fail) {
          ok = false;
          break;
        }
      } else if (!got_u) {
        ok = false;
        break;
      }
      if (u < 0) break;
      const BpUnit w = bp_decode<CAUSAL>(u, p, G);
      for (int it = 0; it < (DQ ? w.T : 0); ++it, ++g) {
        const int hq = w.hkv * G + it / w.nq;
        const int q0 = 64 * (w.qb0 + it % w.nq);
        const bool got = __all_sync(FULL, mbar_wait(dq_full(g & 1), (g >> 1) & 1, abort_flag, lim));
        uint32_t v[64];
        if (got) {
          tc_fence_after();
          const uint32_t dq_tm = tbase + lane_off + C::T_S + 64u * (g & 1);
          tmem_ld32(dq_tm, v);
          tmem_ld32(dq_tm + 32u, v + 32);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(dq_free);
        }
        if constexpr (!C::DQ_TMA) {
          if (!got) {
            ok = false;
            break;
          }
          float* dst = p.dq_acc + (static_cast<long long>(w.b * p.Hq + hq) * p.Npad + q0) * D + r;
#pragma unroll
          for (int c = 0; c < 64; ++c) red_add_f32(dst + c * D, __uint_as_float(v[c]));
        } else {
          if (!got && lane == 0) *dq_fail = 1;
          if (r == 0) bulk_wait_group_read0();  // the previous reduction has read the tile
          named_bar_sync_n(1, 128);
          if (*dq_fail) {
            ok = false;
            break;
          }
          if (r < D) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint8_t* rowp = smem + C::OFF_DQS + hh * C::DQ_HALF + r * 128;
#pragma unroll
              for (int uu = 0; uu < 8; ++uu)
                *reinterpret_cast<uint4*>(rowp + ((uu ^ (r & 7)) * 16)) =
                    make_uint4(v[32 * hh + 4 * uu], v[32 * hh + 4 * uu + 1], v[32 * hh + 4 * uu + 2],
                               v[32 * hh + 4 * uu + 3]);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync_n(1, 128);
          if (r == 0) {
            const int bh = w.b * p.Hq + hq;
            tma_reduce_add_3d(&p.tm_dq, sbase + C::OFF_DQS, q0, 0, bh);
            tma_reduce_add_3d(&p.tm_dq, sbase + C::OFF_DQS + C::DQ_HALF, q0 + 32, 0, bh);
            bulk_commit_group();
          }
        }
      }
      if (!ok) break;
      // the next queue entry: whether another unit (and so V(n + 1)) follows
      int u_next = -1;
      got_u = pop(n + 1, u_next, lane == 0);
      // ---- epilogue: scale * dK into the unit's K buffer (no product reads it any more: its
      // last reader, dQ^T of the unit's last step, completed before dq_full above; without
      // the dQ path before acc_done), dV into the V buffer once V(n + 1) has been copied
      // into TMEM, both in the layout of the K / V loads; each warp stores its 32 key rows
      // with one TMA store per 64 columns (clipped at N) and releases both buffers to the
      // producer once the stores have read them
      const bool got_acc = __all_sync(FULL, mbar_wait(acc_done, n & 1, abort_flag, lim) &&
                                                (u_next < 0 || mbar_wait(v_tmem, (n + 1) & 1, abort_flag, lim)));
      if (!got_acc || !got_u) {
        if (C::DQ_TMA && DQ) {
          if (lane == 0) *dq_fail = 1;  // the next unit's barrier takes all four warps out
          continue;
        }
        ok = false;
        break;
      }
      tc_fence_after();
      const int kb = n & 1;
      const int row0 = 32 * (warp & 3);
      uint8_t* stage_k = smem + C::OFF_K + kb * C::KV_TILE;
      uint8_t* stage_v = smem + C::OFF_V;
      const bool store = w.k0 + row0 < p.N;  // else every row of this warp's box lies past N
      bp_stage_rows<D, BF16, true>(tbase + lane_off + C::T_DK, p.scale, stage_k, r);
      bp_stage_rows<D, BF16, false>(tbase + lane_off + C::T_DV, 1.0f, stage_v, r);
      // both accumulators are in shared memory: the next unit's first gradient products
      // may overwrite them
      tc_fence_before();
      mbar_arrive(acc_free);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (store) {
          for (int ch = 0; ch < C::CHUNKS; ++ch) {
            tma_store_4d(&p.tm_dk, smem_u32(stage_k + ch * C::KV_CHUNK + row0 * 128), ch * 64, w.hkv, w.k0 + row0,
                         w.b);
            tma_store_4d(&p.tm_dv, smem_u32(stage_v + ch * C::KV_CHUNK + row0 * 128), ch * 64, w.hkv, w.k0 + row0,
                         w.b);
          }
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        mbar_arrive(k_empty(kb));
        mbar_arrive(v_empty);
      }
      __syncwarp();
      u = u_next;
    }
    if (C::DQ_TMA && DQ && r == 0) bulk_wait_group0();
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL, bool DQ>
static cudaError_t launch_bwd_persistent_t(const BwdParams& p, cudaStream_t stream) {
  using C = BpCfg<D>;
  const cudaError_t e = prepare_launch_once<fa_bwd_persistent<D, BF16, CAUSAL, DQ>>(C::SMEM, C::THREADS, C::REG_SPLIT);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>((p.N + 127) / 128) * p.B * p.Hkv;
  if (units <= 0) return cudaSuccess;
  unsigned* sched = scheduler_slot();
  if (!sched) return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int grid = static_cast<int>(units < sms ? units : sms);
  fa_bwd_persistent<D, BF16, CAUSAL, DQ><<<grid, C::THREADS, C::SMEM, stream>>>(p, sched, static_cast<int>(units));
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_bwd_persistent_d(const BwdParams& p, bool causal, bool dq, cudaStream_t stream) {
  if (causal)
    return dq ? launch_bwd_persistent_t<D, BF16, true, true>(p, stream)
              : launch_bwd_persistent_t<D, BF16, true, false>(p, stream);
  return dq ? launch_bwd_persistent_t<D, BF16, false, true>(p, stream)
            : launch_bwd_persistent_t<D, BF16, false, false>(p, stream);
}

cudaError_t launch_bwd_persistent(const BwdParams& p, int d, bool bf16, bool causal, bool dq, cudaStream_t stream) {
  if (d == 128)
    return bf16 ? launch_bwd_persistent_d<128, true>(p, causal, dq, stream)
                : launch_bwd_persistent_d<128, false>(p, causal, dq, stream);
  return bf16 ? launch_bwd_persistent_d<64, true>(p, causal, dq, stream)
              : launch_bwd_persistent_d<64, false>(p, causal, dq, stream);
}

}  // namespace fa
