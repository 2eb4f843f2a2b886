// Persistent forward for short sequences: one CTA per SM takes (batch, head, 256-query)
// units from a device-wide counter until none is left.
//
// Method: the same exact attention as the one-CTA-per-unit forward ("FlashAttention-2:
// atención eficiente en GPU para contextos largos", sections "Bloques pequeños,
// normalización global" and "Tres mejoras en la utilización de la GPU", second point:
// the work is split over the sequence as well as batch and heads so the GPU stays full).
// With few key blocks per unit, a CTA that owns one unit spends about as long starting
// (barrier set-up, TMEM allocation, waiting for Q and the first K) and finishing (the
// last P V, reading O out, storing it) as computing.  Here a CTA lives for many units
// and overlaps those phases with its neighbours' work:
//  * warp 8 takes the next unit (one atomic add on the launch's counter) and passes its
//    index to the other roles through a two-entry queue in shared memory; it loads the
//    next unit's Q_t into tile t's buffer as soon as the last S_t of the current unit has
//    been computed, and streams K / V through one ring that runs on across units;
//  * warp 9 issues S_t(next, 0) as soon as that Q_t and K_0 are in, while the softmax
//    warpgroups are still writing out the current unit;
//  * each softmax warpgroup reads O_t out of TMEM, tells the MMA warp that O_t is free,
//    and only then writes O / l and lse to memory from registers (no staging buffer, so
//    nothing in shared memory waits for the stores).
// Units are taken in the same order as the one-CTA-per-unit grid (heaviest first with
// the causal mask), so the dynamic counter balances the tail the way the hardware block
// scheduler does.  The counter pair {next, done} is picked per launch from a small ring
// by the host; the last CTA to finish resets it for the next launch that picks it.
#include "fa_internal.h"
#include "fa_math.cuh"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

namespace fa {

__device__ unsigned g_fa_sched[kSchedSlots][2];

unsigned* scheduler_slot() {
  static std::atomic<unsigned*> base[kMaxSchedDevices];
  static std::atomic<unsigned> next{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSchedDevices) return nullptr;
  unsigned* b = base[dev].load(std::memory_order_acquire);
  if (!b) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_fa_sched) != cudaSuccess) return nullptr;
    b = static_cast<unsigned*>(addr);
    base[dev].store(b, std::memory_order_release);
  }
  return b + 2 * (next.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
}

template <int D>
struct PfCfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  static constexpr int THREADS = 384;
  static constexpr int REG_CTRL = 80, REG_SOFTMAX = 208;
  static constexpr int REG_SPLIT = 128 * REG_CTRL + 256 * REG_SOFTMAX;
  static_assert(REG_SPLIT <= 384 * 168, "register split above the launch allocation");
  // barriers, two of each (one per tile or queue entry): q_full, q_empty, s_full, p_full,
  // o_done, o_free, uq_full, uq_empty; then final; then the ring's full / empty
  static constexpr int B_QF = 0, B_QE = 2, B_SF = 4, B_PF = 6, B_OD = 8, B_OF = 10, B_UF = 12, B_UE = 14,
                       B_FIN = 16, B_KV = 17;
  static constexpr int NBARS = 17 + 2 * STAGES;
  static constexpr int SMEM = 1024 + 2 * TILE_BYTES + STAGES * TILE_BYTES + 8 * NBARS + 64;
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr uint32_t TMEM_COLS = 512;  // S_0, S_1 (128 each), O_0, O_1 (D each)
};

// One unit: 256 queries [256 qb, 256 qb + 256) of (b, h); tile t = rows 256 qb + 128 t,
// visiting n_t key blocks (0 when the tile starts past N).
struct PfUnit {
  int b, h, hkv, qb, n0, n1;
};

template <bool CAUSAL>
__device__ __forceinline__ PfUnit pf_decode(int u, const FwdParams& p) {
  const int nqb = (p.N + 255) / 256;
  const int BH = p.B * p.Hq;
  PfUnit w;
  int bh;
  if (CAUSAL) {
    w.qb = nqb - 1 - u / BH;
    bh = u % BH;
  } else {
    w.qb = u % nqb;
    bh = u / nqb;
  }
  w.h = bh % p.Hq;
  w.b = bh / p.Hq;
  w.hkv = w.h / (p.Hq / p.Hkv);
  auto nb = [&](int r0) { return r0 >= p.N ? 0 : (CAUSAL ? r0 / 128 + 1 : (p.N + 127) / 128); };
  w.n0 = nb(256 * w.qb);
  w.n1 = nb(256 * w.qb + 128);
  return w;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1) fa_fwd_persistent(const __grid_constant__ FwdParams p, unsigned* sched,
                                                            int units) {
  using C = PfCfg<D>;
  extern __shared__ uint8_t smem_raw_pf[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_pf) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * C::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::STAGES * C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* uq = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2] unit queue

  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int base, int i) { return bar0 + 8u * (base + i); };
  auto kv_full = [&](int s) { return bar0 + 8u * (C::B_KV + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (C::B_KV + C::STAGES + s); };
  const uint32_t final_bar = bar(C::B_FIN, 0);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = p.N;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_QF, i), 1);
      mbar_init(bar(C::B_QE, i), 1);
      mbar_init(bar(C::B_SF, i), 1);
      mbar_init(bar(C::B_PF, i), 128);
      mbar_init(bar(C::B_OD, i), 1);
      mbar_init(bar(C::B_OF, i), 128);
      mbar_init(bar(C::B_UF, i), 1);
      mbar_init(bar(C::B_UE, i), 1 + 256);  // the MMA warp's leader and every softmax thread
    }
    mbar_init(final_bar, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
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
  constexpr unsigned FULL = 0xffffffffu;

  if (warp >= 8) {
    setmaxnreg_dec<C::REG_CTRL>();
    const bool leader = elect_one();
    if (warp == 8) {
      // ------------------------------------------------- scheduler + TMA producer
      const int lead_lane = __ffs(__ballot_sync(FULL, leader)) - 1;
      if (leader) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
      }
      bool ok = true;
      int it = 0, c = 0;
      int qcnt[2] = {0, 0};
      auto fetch = [&]() {
        int v = 0;
        if (leader) v = static_cast<int>(atomicAdd(sched, 1u));
        v = __shfl_sync(FULL, v, lead_lane);
        return v < units ? v : -1;
      };
      for (;;) {
        const int u = fetch();
        const int slot = it & 1;
        if (it >= 2 && !__all_sync(FULL, mbar_wait(bar(C::B_UE, slot), ((it >> 1) - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (leader) {
          uq[slot] = u;
          mbar_arrive(bar(C::B_UF, slot));
        }
        ++it;
        if (u < 0) break;
        const PfUnit w = pf_decode<CAUSAL>(u, p);
        for (int t = 0; t < 2 && ok; ++t) {
          if ((t ? w.n1 : w.n0) == 0) continue;
          // Q_t's buffer is free once the previous unit's last S_t has been computed
          if (qcnt[t] > 0 &&
              !__all_sync(FULL, mbar_wait(bar(C::B_QE, t), (qcnt[t] - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(bar(C::B_QF, t), C::TILE_BYTES);
            for (int ch = 0; ch < C::CHUNKS; ++ch)
              tma_load_4d(smem_u32(sQ + t * C::TILE_BYTES + ch * C::CHUNK_BYTES), &p.tm_q, bar(C::B_QF, t), ch * 64,
                          w.h, 256 * w.qb + 128 * t, w.b);
          }
          ++qcnt[t];
        }
        if (!ok) break;
        const int nmax = w.n0 > w.n1 ? w.n0 : w.n1;
        for (int j = 0; j < nmax && ok; ++j) {
          for (int kind = 0; kind < 2; ++kind, ++c) {
            const int s = c % C::STAGES;
            if (c >= C::STAGES &&
                !__all_sync(FULL, mbar_wait(kv_empty(s), ((c / C::STAGES) - 1) & 1, abort_flag, lim))) {
              ok = false;
              break;
            }
            if (leader) {
              mbar_arrive_expect_tx(kv_full(s), C::TILE_BYTES);
              const CUtensorMap* map = kind ? &p.tm_v : &p.tm_k;
              for (int ch = 0; ch < C::CHUNKS; ++ch)
                tma_load_4d(smem_u32(sKV + s * C::TILE_BYTES + ch * C::CHUNK_BYTES), map, kv_full(s), ch * 64, w.hkv,
                            128 * j, w.b);
            }
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        if (leader) fail();
        // let the copies in flight land before the CTA's shared memory goes away
        for (int i = (c > C::STAGES ? c - C::STAGES : 0); i < c; ++i)
          mbar_wait(kv_full(i % C::STAGES), (i / C::STAGES) & 1, no_abort, lim);
        for (int t = 0; t < 2; ++t)
          if (qcnt[t] > 0) mbar_wait(bar(C::B_QF, t), (qcnt[t] - 1) & 1, no_abort, lim);
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
    } else if (warp == 9) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t id_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t id_pv = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
      const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
      const uint64_t dq0 = smem_desc_sw128(sq, 16, 1024), dkv0 = smem_desc_sw128(skv, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(skv, C::CHUNK_BYTES, 1024);
      bool ok = true;
      int it = 0, c = 0;
      int cnt[2] = {0, 0};  // units in which tile t took part (Q loads, O rounds)
      int blk[2] = {0, 0};  // key blocks tile t has gone through (S / P rounds)
      for (;;) {
        const int slot = it & 1;
        if (!__all_sync(FULL, mbar_wait(bar(C::B_UF, slot), (it >> 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        const int u = uq[slot];
        __syncwarp();
        if (leader) mbar_arrive(bar(C::B_UE, slot));
        ++it;
        if (u < 0) break;
        const PfUnit w = pf_decode<CAUSAL>(u, p);
        const int nmax = w.n0 > w.n1 ? w.n0 : w.n1;
        for (int j = 0; j <= nmax && ok; ++j) {
          const int kc = c + 2 * j, vc = c + 2 * j - 1;
          const int kslot = kc % C::STAGES, vslot = vc % C::STAGES;
          if (j < nmax && !__all_sync(FULL, mbar_wait(kv_full(kslot), (kc / C::STAGES) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (j > 0 && !__all_sync(FULL, mbar_wait(kv_full(vslot), (vc / C::STAGES) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int t = 0; t < 2; ++t) {
            const int nt = t ? w.n1 : w.n0;
            const uint32_t s_tm = tbase + 128u * t;
            const uint32_t o_tm = tbase + 256u + uint32_t(D) * t;
            if (j > 0 && j - 1 < nt) {
              // O_t (+)= P_t(j-1) V_{j-1}; the first product of a unit overwrites O_t, which
              // the softmax warpgroup must have read out for the previous unit
              bool w_ok = mbar_wait(bar(C::B_PF, t), (blk[t] + j - 1) & 1, abort_flag, lim);
              if (j == 1 && cnt[t] > 0) w_ok = w_ok && mbar_wait(bar(C::B_OF, t), (cnt[t] - 1) & 1, abort_flag, lim);
              if (!__all_sync(FULL, w_ok)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t vd = dv0 + static_cast<uint64_t>((vslot * C::TILE_BYTES) >> 4);
              if (leader) {
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(o_tm, s_tm + 8u * kk, vd + static_cast<uint64_t>((kk * 2048) >> 4), id_pv,
                         (j - 1 > 0 || kk > 0) ? 1u : 0u);
                if (j == nt) mma_commit(bar(C::B_OD, t));
              }
            }
            if (j < nt) {
              // S_t = Q_t K_j^T, both K-major
              if (j == 0) {
                if (!__all_sync(FULL, mbar_wait(bar(C::B_QF, t), cnt[t] & 1, abort_flag, lim))) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              const uint64_t qd = dq0 + static_cast<uint64_t>((t * C::TILE_BYTES) >> 4);
              const uint64_t kd = dkv0 + static_cast<uint64_t>((kslot * C::TILE_BYTES) >> 4);
              if (leader) {
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint64_t off = static_cast<uint64_t>(((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32) >> 4);
                  mma_ss(s_tm, qd + off, kd + off, id_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::B_SF, t));
                if (j == nt - 1) mma_commit(bar(C::B_QE, t));  // Q_t may be reloaded
              }
            }
          }
          if (!ok) break;
          if (leader) {
            if (j > 0) mma_commit(kv_empty(vslot));
            if (j < nmax) mma_commit(kv_empty(kslot));
          }
        }
        if (!ok) break;
        c += 2 * nmax;
        for (int t = 0; t < 2; ++t) {
          const int nt = t ? w.n1 : w.n0;
          if (nt > 0) {
            ++cnt[t];
            blk[t] += nt;
          }
        }
      }
      if (!ok && leader) fail();
      if (leader) mma_commit(final_bar);
      mbar_wait(final_bar, 0, no_abort, lim);
      // the last commits to kv_empty and q_empty have no consumer: let them land first
      if (ok) {
        for (int i = (c > C::STAGES ? c - C::STAGES : 0); i < c; ++i)
          mbar_wait(kv_empty(i % C::STAGES), (i / C::STAGES) & 1, no_abort, lim);
        for (int t = 0; t < 2; ++t)
          if (cnt[t] > 0) mbar_wait(bar(C::B_QE, t), (cnt[t] - 1) & 1, no_abort, lim);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<C::REG_SOFTMAX>();
    // ----------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;
    const int rit = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t s_tm = tbase + lane_off + 128u * t;
    const uint32_t o_tm = tbase + lane_off + 256u + uint32_t(D) * t;
    const float cl2 = p.scale_log2;
    bool ok = true;
    int it = 0, cnt = 0, blk = 0;
    for (;;) {
      const int slot = it & 1;
      if (!__all_sync(FULL, mbar_wait(bar(C::B_UF, slot), (it >> 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      const int u = uq[slot];
      mbar_arrive(bar(C::B_UE, slot));
      ++it;
      if (u < 0) break;
      const PfUnit w = pf_decode<CAUSAL>(u, p);
      const int nt = t ? w.n1 : w.n0;
      if (nt == 0) continue;
      const int row = 256 * w.qb + 128 * t + rit;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        if (!__all_sync(FULL, mbar_wait(bar(C::B_SF, t), (blk + j) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_tm + 32u * cc, sr + 32 * cc);
        tmem_wait_ld();
        float* s = reinterpret_cast<float*>(sr);
        if (j == nt - 1 && (CAUSAL || (N & 127))) {
          const int nvis = (CAUSAL ? min(N, row + 1) : N) - 128 * j;
#pragma unroll
          for (int cc = 0; cc < 128; ++cc)
            if (cc >= nvis) s[cc] = -INFINITY;
        }
        const float mx = rowmax128(s);
        if (j == 0) {
          m = mx;
        } else if (__any_sync(FULL, (mx - m) * cl2 > 8.0f)) {
          // lazy correction of O_t and l (PV_t(j-1) is complete: S_t(j) was issued after it)
          const float m_new = fmaxf(m, mx);
          const float alpha = ex2_mufu((m - m_new) * cl2);
          m = m_new;
          l *= alpha;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32(o_tm + 32u * cc, orr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(o_tm + 32u * cc, orr);
          }
          tmem_wait_st();
        }
        const float neg = -m * cl2;
        const uint64_t cl2x2 = f2pack(cl2, cl2), negx2 = f2pack(neg, neg);
        uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
        for (int cc = 0; cc < 128; cc += 4) {
          float a0, a1, a2, a3;
          f2unpack(ffma2(f2pack(s[cc], s[cc + 1]), cl2x2, negx2), a0, a1);
          f2unpack(ffma2(f2pack(s[cc + 2], s[cc + 3]), cl2x2, negx2), a2, a3);
          s[cc] = ex2_mufu(a0);
          s[cc + 1] = ex2_mufu(a1);
          s[cc + 2] = ex2_mufu(a2);
          s[cc + 3] = ex2_mufu(a3);
          acc0 = fadd2(acc0, f2pack(s[cc], s[cc + 1]));
          acc1 = fadd2(acc1, f2pack(s[cc + 2], s[cc + 3]));
        }
        float sa, sb, sc2, sd;
        f2unpack(acc0, sa, sb);
        f2unpack(acc1, sc2, sd);
        l += (sa + sb) + (sc2 + sd);
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) pk[i] = pack_half2<BF16>(s[2 * i], s[2 * i + 1]);
        tmem_st32(s_tm, pk);
        tmem_st32(s_tm + 32u, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::B_PF, t));
      }
      if (!ok) break;
      blk += nt;
      if (!__all_sync(FULL, mbar_wait(bar(C::B_OD, t), cnt & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      ++cnt;
      tc_fence_after();
      // ---- epilogue: O_t out of TMEM (then O_t is free for the next unit), O / l rounded to
      // 16 bits and stored row by row, lse = scale * m + ln l
      const float inv = 1.0f / l;
      uint32_t pk[D / 2];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t orr[32];
        tmem_ld32(o_tm + 32u * cc, orr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[16 * cc + i] = pack_half2<BF16>(__uint_as_float(orr[2 * i]) * inv, __uint_as_float(orr[2 * i + 1]) * inv);
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_OF, t));
      if (row < N) {
        uint16_t* orow = p.o + ((static_cast<long long>(w.b) * N + row) * p.Hq + w.h) * D;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          *reinterpret_cast<uint4*>(orow + 8 * i) = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        p.lse[(static_cast<size_t>(w.b) * p.Hq + w.h) * N + row] = m * p.scale + logf(l);
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_fwd_persistent_t(const FwdParams& p, cudaStream_t stream) {
  using C = PfCfg<D>;
  cudaError_t e = prepare_launch_once<fa_fwd_persistent<D, BF16, CAUSAL>>(C::SMEM, C::THREADS, C::REG_SPLIT);
  if (e != cudaSuccess) return e;
  unsigned* sched = scheduler_slot();
  if (!sched) return cudaErrorInvalidValue;
  const long long units = static_cast<long long>((p.N + 255) / 256) * p.B * p.Hq;
  const int sms = device_sm_count();
  const int grid = static_cast<int>(units < sms ? units : sms);
  fa_fwd_persistent<D, BF16, CAUSAL><<<grid, C::THREADS, C::SMEM, stream>>>(p, sched, static_cast<int>(units));
  return cudaGetLastError();
}

cudaError_t launch_fwd_persistent(const FwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream) {
  const bool bf = dtype == FA_BF16;
  if (d == 128) {
    if (bf) return causal ? launch_fwd_persistent_t<128, true, true>(p, stream)
                          : launch_fwd_persistent_t<128, true, false>(p, stream);
    return causal ? launch_fwd_persistent_t<128, false, true>(p, stream)
                  : launch_fwd_persistent_t<128, false, false>(p, stream);
  }
  if (bf) return causal ? launch_fwd_persistent_t<64, true, true>(p, stream)
                        : launch_fwd_persistent_t<64, true, false>(p, stream);
  return causal ? launch_fwd_persistent_t<64, false, true>(p, stream)
                : launch_fwd_persistent_t<64, false, false>(p, stream);
}

}  // namespace fa
