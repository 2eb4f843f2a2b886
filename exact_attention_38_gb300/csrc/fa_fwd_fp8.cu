// FP8 (E4M3) forward of exact attention on sm_103a.
//
// The pages report an 8-bit forward as the fastest mode ("FlashAttention-T:
// Optimización GPU para LLMs Escalables", section "Innovaciones técnicas frente a
// FlashAttention original"); the method is still the tiled exact attention of
// "FlashAttention-2: atención eficiente en GPU para contextos largos" (section "Bloques
// pequeños, normalización global"), only with 8-bit operands for the two products.
//
// Inputs q, k, v are E4M3 with one descale factor per tensor (real value = stored value
// x descale).  The score scale folds the softmax scale and both descales; P is scaled
// by 2^7 before its E4M3 rounding, so that values down to about 2^-16 of the row's
// largest keep a representable step.  With the running maximum allowed to lag by tau in
// log2 units, the scaled values reach 2^(7 + tau), which must stay below E4M3's 448:
// tau = 1.5 (the 16-bit kernel's 8 would saturate).  The 2^7 is added to the exponent,
// and the row sum l carries it too, so O / l needs no extra factor; O is multiplied by
// v's descale and written in bf16, lse (fp32) subtracts 7 ln 2.
//
// The pair (2^7, 1.5) was measured against (2^8, 0.5): the smaller lag bound made
// about a quarter of the blocks rescale O at 16k keys (any row of a warp triggers the
// warp's 128-column TMEM rescale), against about one in twelve, and the kernel ran 7%
// slower.
//
// GB300 form: the 16-bit forward's pipeline (two 128-row query tiles per CTA, a TMA
// warp, an MMA warp, one softmax warpgroup per tile, P from tensor memory) with
// tcgen05.mma.kind::f8f6f4 products, K = 32 per instruction.  Both operands of an 8-bit
// product are kept K-major: S = Q K^T reads Q and K as stored, and O += P V reads a
// transposed copy V^T [B*Hkv, d, Npad] that a small kernel writes first (one extra pass
// over V, 2 bytes per element).  Head dimension 128.
#include "fa_internal.h"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>

namespace fa {

namespace {

constexpr int kD = 128;
constexpr int kTile = 128 * 128;  // Q, K or V^T tile: 128 rows x 128 bytes
constexpr int kStages = 8;        // K / V^T ring
constexpr int kThreads = 384;
constexpr int kNbars = 8 + 2 * kStages + 1;
constexpr int kSmem = 1024 + 2 * kTile + kStages * kTile + 8 * kNbars + 64;
constexpr float kLn2 = 0.69314718055994531f;
// P is rounded to E4M3 as P * 2^kPScaleLog2.
constexpr float kPScaleLog2 = 7.0f;
// Lazy rescale threshold (log2 units).  With a stale maximum p can reach 2^tau, so
// 2^kPScaleLog2 * 2^tau must stay below E4M3's largest value 448: 2^8.5 = 362.
constexpr float kTau = 1.5f;
static_assert(kPScaleLog2 + kTau <= 8.5f, "scaled P must stay below E4M3's 448");
static_assert(kSmem <= 232448, "shared memory budget");

__device__ __forceinline__ float f8_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four values -> four E4M3 bytes (round to nearest, saturating), element 0 in the low byte.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace

// V [B, N, Hkv, 128] -> V^T [B*Hkv, 128, Npad] (keys contiguous), zero past N.  One CTA
// per (b*Hkv + h, 128-key tile): rows read as 128-byte lines, the tile turned through
// shared memory, written as 128-byte lines.
__global__ void __launch_bounds__(256) fa_fp8_transpose_v(const __grid_constant__ Fp8Params p) {
  __shared__ uint8_t tile[128][132];
  const int ntiles = p.Npad / 128;
  const int bh = static_cast<int>(blockIdx.x / ntiles);
  const int n0 = 128 * static_cast<int>(blockIdx.x % ntiles);
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  for (int i = threadIdx.x; i < 128 * 8; i += 256) {  // 16 bytes per thread and step
    const int k = i >> 3, part = i & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n0 + k < p.N)
      v = *reinterpret_cast<const uint4*>(p.v + ((static_cast<long long>(b) * p.N + n0 + k) * p.Hkv + h) * kD +
                                          16 * part);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) *reinterpret_cast<uint32_t*>(&tile[k][16 * part + 4 * u]) = w[u];
  }
  __syncthreads();
  uint8_t* dst = p.vt + static_cast<long long>(bh) * kD * p.Npad + n0;
  for (int i = threadIdx.x; i < 128 * 32; i += 256) {  // 4 keys of one dimension per step
    const int dd = i >> 5, k4 = (i & 31) * 4;
    const uint32_t w = tile[k4][dd] | (tile[k4 + 1][dd] << 8) | (tile[k4 + 2][dd] << 16) |
                       (static_cast<uint32_t>(tile[k4 + 3][dd]) << 24);
    *reinterpret_cast<uint32_t*>(dst + static_cast<long long>(dd) * p.Npad + k4) = w;
  }
}

template <bool CAUSAL, bool BLOCK>
__global__ void __launch_bounds__(384, 1) fa_fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
  extern __shared__ uint8_t smem_raw_f8[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_f8) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * kTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + kStages * kTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNbars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]

  const uint32_t bar0 = smem_u32(bars);
  auto q_full = [&](int t) { return bar0 + 8u * (0 + t); };
  auto s_full = [&](int t) { return bar0 + 8u * (2 + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (4 + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (6 + t); };
  auto kv_full = [&](int st) { return bar0 + 8u * (8 + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (8 + kStages + st); };
  const uint32_t final_bar = bar0 + 8u * (8 + 2 * kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work decode (as the 16-bit forward): 256 query rows of one (batch, head) per
  // CTA; without the mask the query blocks of a head are consecutive CTAs, with it the
  // heaviest blocks go first
  const int N = p.N;
  const int nqb = (N + 255) / 256;
  const int BH = p.B * p.Hq;
  int qb, bh;
  if (CAUSAL) {
    qb = nqb - 1 - static_cast<int>(blockIdx.x / BH);
    bh = static_cast<int>(blockIdx.x % BH);
  } else {
    qb = static_cast<int>(blockIdx.x % nqb);
    bh = static_cast<int>(blockIdx.x / nqb);
  }
  const int h = bh % p.Hq, b = bh / p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  const int nkb = (N + 127) / 128;
  const int r00 = qb * 256, r01 = qb * 256 + 128;
  const int n0 = CAUSAL ? (r00 / 128 + 1) : nkb;
  const int n1 = (r01 >= N) ? 0 : (CAUSAL ? (r01 / 128 + 1) : nkb);
  auto n_of = [&](int t) { return t ? n1 : n0; };
  auto r0_of = [&](int t) { return t ? r01 : r00; };
  const int nmax = n0 > n1 ? n0 : n1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    wg_fail[0] = wg_fail[1] = 0;
    for (int i = 0; i < 8; ++i) mbar_init(bar0 + 8u * i, (i >= 4 && i < 6) ? 128u : 1u);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
    }
    mbar_init(final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.err, kDevErrTimeout);
  };
  constexpr unsigned FULL = 0xffffffffu;

  if (warp >= 8) {
    setmaxnreg_dec<80>();
    const bool leader = elect_one();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (leader) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_vt);
        for (int t = 0; t < 2; ++t) {
          if (n_of(t) == 0) continue;
          mbar_arrive_expect_tx(q_full(t), kTile);
          tma_load_4d(smem_u32(sQ + t * kTile), &p.tm_q, q_full(t), 0, h, r0_of(t), b);
        }
      }
      int c = 0;
      bool ok = true;
      for (int j = 0; j < nmax && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind, ++c) {  // K_j, then V_j^T
          const int slot = c % kStages;
          if (c >= kStages &&
              !__all_sync(FULL, mbar_wait(kv_empty(slot), ((c / kStages) - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(kv_full(slot), kTile);
            const uint32_t dst = smem_u32(sKV + slot * kTile);
            if (kind == 0)
              tma_load_4d(dst, &p.tm_k, kv_full(slot), 0, hkv, 128 * j, b);
            else
              tma_load_3d(dst, &p.tm_vt, kv_full(slot), 128 * j, 0, b * p.Hkv + hkv);
          }
        }
      }
      if (!ok) {
        if (leader) fail();
        for (int i = (c > kStages ? c - kStages : 0); i < c; ++i)
          mbar_wait(kv_full(i % kStages), (i / kStages) & 1, nullptr, lim);
        for (int t = 0; t < 2; ++t)
          if (n_of(t)) mbar_wait(q_full(t), 0, nullptr, lim);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t id_qk = idesc_e4m3(128, 128);
      constexpr uint32_t id_pv = idesc_e4m3(128, kD);
      bool ok = true;
      for (int t = 0; t < 2 && ok; ++t)
        if (n_of(t)) ok = __all_sync(FULL, mbar_wait(q_full(t), 0, abort_flag, lim));
      // K-major, 128-byte swizzle: one 128-byte row per element row; a K = 32 step of an
      // 8-bit product advances 32 bytes inside the row
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dkv0 = smem_desc_sw128(smem_u32(sKV), 16, 1024);
      for (int j = 0; j <= nmax && ok; ++j) {
        const int kc = 2 * j, vc = 2 * j - 1;
        const int kslot = kc % kStages, vslot = (vc + kStages) % kStages;
        if (j < nmax && !__all_sync(FULL, mbar_wait(kv_full(kslot), (kc / kStages) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (j > 0 && !__all_sync(FULL, mbar_wait(kv_full(vslot), (vc / kStages) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          const uint32_t s_tm = tbase + 128u * t;
          const uint32_t o_tm = tbase + 256u + uint32_t(kD) * t;
          if (j > 0 && j - 1 < n_of(t)) {
            // O_t += P_t(j-1) V_{j-1}: P from TMEM (four E4M3 per column over S_t's first
            // 32 columns), V^T K-major
            if (!__all_sync(FULL, mbar_wait(p_full(t), (j - 1) & 1, abort_flag, lim))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = dkv0 + static_cast<uint64_t>((vslot * kTile) >> 4);
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts_f8(o_tm, s_tm + 8u * kk, vd + static_cast<uint64_t>((kk * 32) >> 4), id_pv,
                          (j - 1 > 0 || kk > 0) ? 1u : 0u);
              if (j - 1 == n_of(t) - 1) mma_commit(o_done(t));
            }
          }
          if (j < n_of(t)) {
            // S_t = Q_t K_j^T
            const uint64_t qd = dq0 + static_cast<uint64_t>((t * kTile) >> 4);
            const uint64_t kd = dkv0 + static_cast<uint64_t>((kslot * kTile) >> 4);
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss_f8(s_tm, qd + static_cast<uint64_t>((kk * 32) >> 4), kd + static_cast<uint64_t>((kk * 32) >> 4),
                          id_qk, kk > 0 ? 1u : 0u);
              mma_commit(s_full(t));
            }
          }
        }
        if (!ok) break;
        if (leader) {
          if (j > 0) mma_commit(kv_empty(vslot));
          if (j < nmax) mma_commit(kv_empty(kslot));
        }
      }
      if (!ok && leader) fail();
      if (leader) mma_commit(final_bar);
      mbar_wait(final_bar, 0, nullptr, lim);
      if (ok) {
        for (int c = (2 * nmax > kStages ? 2 * nmax - kStages : 0); c < 2 * nmax; ++c)
          mbar_wait(kv_empty(c % kStages), (c / kStages) & 1, nullptr, lim);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<208>();
    // ----------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;
    const int rit = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t s_tm = tbase + lane_off + 128u * t;
    const uint32_t o_tm = tbase + lane_off + 256u + uint32_t(kD) * t;
    const float cl2 = p.score_log2;
    const int row = r0_of(t) + rit;
    float m = -INFINITY, l = 0.f;
    // Per-block descales: the score multiplier changes from key block to key block, so m is
    // kept in log2 units of the scaled score (not of the raw product), and V's descale of
    // block j enters P's exponent as log2(v_j / v_max) <= 0, v_max the largest over the
    // tile's blocks: P * 2^7 * v_j / v_max still fits E4M3, l sums P without that factor
    // (its block sum is divided by v_j / v_max), and O / l is multiplied by v_max.
    float q_ds = 0.f, v_max = 0.f, v_inv = 0.f, k_next = 0.f, v_next = 0.f;
    const int kvb = BLOCK ? (b * p.Hkv + hkv) * p.nb : 0;  // this head's first block descale
    if constexpr (BLOCK) {
      if (n_of(t) > 0) {
        q_ds = p.q_bs[(b * p.Hq + h) * p.nb + (r0_of(t) >> 7)];
        for (int j = lane; j < n_of(t); j += 32) v_max = fmaxf(v_max, p.v_bs[kvb + j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v_max = fmaxf(v_max, __shfl_xor_sync(FULL, v_max, o));
        v_inv = 1.0f / v_max;
        k_next = p.k_bs[kvb];  // block j's descales are read one block ahead
        v_next = p.v_bs[kvb];
      }
    }
    bool ok = true;
    for (int j = 0; j < n_of(t); ++j) {
      if (!__all_sync(FULL, mbar_wait(s_full(t), j & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + 32u * c, sr + 32 * c);
      tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sr);
      if (j == n_of(t) - 1 && (CAUSAL || (N & 127))) {
        const int k0 = 128 * j;
        const int nvis = CAUSAL ? min(N, row + 1) - k0 : N - k0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= nvis) s[c] = -INFINITY;
      }
      // score multiplier to log2 units; with per-block descales m is held in those units
      float cj = cl2, vr = 1.0f, vr_inv = 1.0f;  // vr = v_j / v_max (per-block descales)
      if constexpr (BLOCK) {
        cj = p.scale_log2 * q_ds * k_next;
        vr = v_next * v_inv;
        vr_inv = __fdividef(v_max, v_next);
        if (j + 1 < n_of(t)) {
          k_next = p.k_bs[kvb + j + 1];
          v_next = p.v_bs[kvb + j + 1];
        }
      }
      const float mx = BLOCK ? rowmax128(s) * cj : rowmax128(s);
      const float mdiff = BLOCK ? 1.0f : cl2;  // log2 units per unit of m
      if (j == 0) {
        m = mx;
      } else if (__any_sync(FULL, (mx - m) * mdiff > kTau)) {
        const float m_new = fmaxf(m, mx);
        const float alpha = f8_ex2((m - m_new) * mdiff);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(o_tm + 32u * c, orr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(o_tm + 32u * c, orr);
        }
        tmem_wait_st();
      }
      // the pre-scale of P is folded into the exponent: p = exp2(s c - m c + 7); l sums
      // the scaled values too, so it cancels in O / l (and lse subtracts 7 ln 2)
      const float neg = BLOCK ? -m + kPScaleLog2 + __log2f(vr) : -m * cl2 + kPScaleLog2;
      const uint64_t cl2x2 = f2pack(cj, cj), negx2 = f2pack(neg, neg);
      uint64_t acc0 = 0ull, acc1 = 0ull;
      uint32_t pk[32];
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) {
        float a0, a1, a2, a3;
        f2unpack(ffma2(f2pack(s[4 * c4], s[4 * c4 + 1]), cl2x2, negx2), a0, a1);
        f2unpack(ffma2(f2pack(s[4 * c4 + 2], s[4 * c4 + 3]), cl2x2, negx2), a2, a3);
        const uint64_t p01 = f2pack(f8_ex2(a0), f8_ex2(a1)), p23 = f2pack(f8_ex2(a2), f8_ex2(a3));
        acc0 = fadd2(acc0, p01);
        acc1 = fadd2(acc1, p23);
        float q0, q1, q2, q3;
        f2unpack(p01, q0, q1);
        f2unpack(p23, q2, q3);
        pk[c4] = pack4_e4m3(q0, q1, q2, q3);
      }
      float sa, sb, sc2, sd;
      f2unpack(acc0, sa, sb);
      f2unpack(acc1, sc2, sd);
      if constexpr (BLOCK)
        l += ((sa + sb) + (sc2 + sd)) * vr_inv;
      else
        l += (sa + sb) + (sc2 + sd);
      tmem_st32(s_tm, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(t));
    }
    if (n_of(t) > 0) {
      if (ok && !mbar_wait(o_done(t), 0, abort_flag, lim)) ok = false;
      if (!ok) {
        wg_fail[t] = 1;
        fail();
      }
      named_bar_sync_n(1 + t, 128);
      if (wg_fail[t] == 0) {
        tc_fence_after();
        const float f = (BLOCK ? v_max : p.out_scale) / l;
        uint16_t* orow = p.o + ((static_cast<long long>(b) * N + row) * p.Hq + h) * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(o_tm + 32u * c, orr);
          tmem_wait_ld();
          if (row >= N) continue;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(orr[8 * u + 0]) * f, __uint_as_float(orr[8 * u + 1]) * f);
            w.y = pack_bf16x2(__uint_as_float(orr[8 * u + 2]) * f, __uint_as_float(orr[8 * u + 3]) * f);
            w.z = pack_bf16x2(__uint_as_float(orr[8 * u + 4]) * f, __uint_as_float(orr[8 * u + 5]) * f);
            w.w = pack_bf16x2(__uint_as_float(orr[8 * u + 6]) * f, __uint_as_float(orr[8 * u + 7]) * f);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * u) = w;
          }
        }
        if (row < N)
          p.lse[(static_cast<size_t>(b) * p.Hq + h) * N + row] =
              (BLOCK ? m * kLn2 : m * p.score_scale) + logf(l) - kPScaleLog2 * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

cudaError_t launch_fwd_fp8(const Fp8Params& p, bool causal, cudaStream_t stream) {
  {
    const long long grid = static_cast<long long>(p.B) * p.Hkv * (p.Npad / 128);
    fa_fp8_transpose_v<<<static_cast<unsigned>(grid), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const bool block = p.q_bs != nullptr;
  auto kern = causal ? (block ? fa_fwd_fp8_kernel<true, true> : fa_fwd_fp8_kernel<true, false>)
                     : (block ? fa_fwd_fp8_kernel<false, true> : fa_fwd_fp8_kernel<false, false>);
  constexpr int kSplit = 128 * 80 + 256 * 208;
  cudaError_t e = causal ? (block ? prepare_launch_once<fa_fwd_fp8_kernel<true, true>>(kSmem, 384, kSplit)
                                  : prepare_launch_once<fa_fwd_fp8_kernel<true, false>>(kSmem, 384, kSplit))
                         : (block ? prepare_launch_once<fa_fwd_fp8_kernel<false, true>>(kSmem, 384, kSplit)
                                  : prepare_launch_once<fa_fwd_fp8_kernel<false, false>>(kSmem, 384, kSplit));
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((p.N + 255) / 256) * p.B * p.Hq;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
