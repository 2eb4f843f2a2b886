// dQ of the backward pass in a fixed summation order (the deterministic backward).
//
// The main backward kernel owns a block of keys and adds its dS K contribution into an
// fp32 dQ accumulator with tensor-memory-access reductions; the order in which CTAs
// land their additions varies from run to run, so dQ's last bits do too.  This kernel
// instead owns a tile of 128 queries and walks the key blocks in ascending order,
// recomputing S = Q K^T and dP = dO V^T and accumulating dQ = scale * sum_j dS_j K_j in
// tensor memory: every dQ element is then summed in the same order on every run.  The
// price is two more GEMM-shaped products per (query, key) block (S and dP are computed
// by both kernels).  The gradient is the closed form of the pages' exact attention
// ("FlashAttention-2: atención eficiente en GPU para contextos largos", section "Bloques
// pequeños, normalización global"): dS = P * (dP - D), P = exp(s - lse).
//
// GB300 form (one 128-query tile per CTA, 384 threads):
//  * warp 8 streams Q and dO once and K_j / V_j through a ring (128-byte swizzle);
//  * warp 9 issues S_j = Q K_j^T into one of two TMEM buffers and dP_j = dO V_j^T, then
//    dQ += dS_{j-1} K_{j-1} with dS read from TMEM, where the dS warpgroups left it as
//    16-bit pairs over S; S double-buffered so S_{j+1} and dP_{j+1} overlap the dS work
//    of block j;
//  * warpgroups 0 and 1 (thread = query row = TMEM lane) each take 64 of the block's 128
//    keys and turn S_j, dP_j into dS = exp2(s * scale * log2 e - lse * log2 e) * (dP - D),
//    written over the columns of S they read (keys 0-63 packed at columns 0-31, keys
//    64-127 at columns 64-95);
//  * epilogue: dQ * scale rounded to 16 bits, stored row by row (each warpgroup half of
//    the head dimension).
#include "fa_internal.h"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

template <int D>
struct DqCfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;  // Q, dO, or one K / V block of 128 rows
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  static constexpr int THREADS = 384;
  // barriers: q_full, s_full[2], dp_free, ds_ready[2], dq_done, final, kv_full[S], kv_empty[S]
  static constexpr int NBARS = 8 + 2 * STAGES;
  static constexpr int SMEM = 1024 + (2 + STAGES) * TILE_BYTES + 8 * NBARS + 64;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM: S / dS buffers [0,128) and [128,256), dP [256,384), dQ [384,384+D)
  static constexpr uint32_t T_S = 0, T_DP = 256, T_DQ = 384, TMEM_COLS = 512;
};

__device__ __forceinline__ float dq_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t dq_pack2(float lo, float hi) {
  uint32_t r;
  if (BF16)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw_dq[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_dq) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + C::TILE_BYTES;
  uint8_t* sKV = smem + 2 * C::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::STAGES * C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0, dp_free = bar0 + 24u, dq_done = bar0 + 48u, final_bar = bar0 + 56u;
  auto s_full = [&](int b) { return bar0 + 8u * (1 + b); };
  auto ds_ready = [&](int b) { return bar0 + 8u * (4 + b); };
  auto kv_full = [&](int st) { return bar0 + 8u * (8 + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (8 + C::STAGES + st); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work decode: CTA = (batch, query head, 128-query tile); with the mask, the
  // tiles with most key blocks first; query heads of a GQA group adjacent
  const int N = p.N;
  const int nqt = (N + 127) / 128;
  const int BH = p.B * p.Hq;
  int qt, bh;
  if (CAUSAL) {
    qt = nqt - 1 - static_cast<int>(blockIdx.x / BH);
    bh = static_cast<int>(blockIdx.x % BH);
  } else {
    qt = static_cast<int>(blockIdx.x % nqt);
    bh = static_cast<int>(blockIdx.x / nqt);
  }
  const int h = bh % p.Hq, b = bh / p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  const int r0 = 128 * qt;
  const int n = CAUSAL ? qt + 1 : (N + 127) / 128;  // key blocks (keys past N are zero rows)

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *wg_fail = 0;
    mbar_init(q_full, 1);
    mbar_init(s_full(0), 1);
    mbar_init(s_full(1), 1);
    mbar_init(dp_free, 256);
    mbar_init(ds_ready(0), 256);
    mbar_init(ds_ready(1), 256);
    mbar_init(dq_done, 1);
    mbar_init(final_bar, 1);
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
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
        tma_prefetch_desc(&p.tm_do);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        // the Q / dO maps have 64-row boxes (the main backward kernel's step): two per
        // 128-row chunk, the second 64 rows (8 KB) further on
        mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
        for (int ch = 0; ch < C::CHUNKS; ++ch) {
          for (int half = 0; half < 2; ++half) {
            const int off = ch * C::CHUNK_BYTES + half * 8192;
            tma_load_4d(smem_u32(sQ + off), &p.tm_q, q_full, ch * 64, h, r0 + 64 * half, b);
            tma_load_4d(smem_u32(sDO + off), &p.tm_do, q_full, ch * 64, h, r0 + 64 * half, b);
          }
        }
      }
      int c = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind, ++c) {  // K_j then V_j
          const int slot = c % C::STAGES;
          if (c >= C::STAGES &&
              !__all_sync(FULL, mbar_wait(kv_empty(slot), ((c / C::STAGES) - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(kv_full(slot), C::TILE_BYTES);
            const CUtensorMap* map = kind ? &p.tm_v : &p.tm_k;
            for (int ch = 0; ch < C::CHUNKS; ++ch)
              tma_load_4d(smem_u32(sKV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES), map, kv_full(slot), ch * 64,
                          hkv, 128 * j, b);
          }
        }
      }
      if (!ok) {
        if (leader) fail();
        for (int i = (c > C::STAGES ? c - C::STAGES : 0); i < c; ++i)
          mbar_wait(kv_full(i % C::STAGES), (i / C::STAGES) & 1, nullptr, lim);
        mbar_wait(q_full, 0, nullptr, lim);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t bf = BF16 ? 1u : 0u;
      constexpr uint32_t id_sq = idesc_f16(128, 128, bf, 0, 0);  // S, dP: both operands K-major
      constexpr uint32_t id_dq = idesc_f16(128, D, bf, 0, 1);    // dQ: K MN-major
      bool ok = __all_sync(FULL, mbar_wait(q_full, 0, abort_flag, lim));
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t ddo0 = smem_desc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t dkv0 = smem_desc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dk_mn0 = smem_desc_sw128(smem_u32(sKV), C::CHUNK_BYTES, 1024);
      auto u16 = [](int bytes) { return static_cast<uint64_t>(bytes >> 4); };
      for (int j = 0; j <= n && ok; ++j) {
        const int kc = 2 * j, vc = 2 * j + 1;
        if (j < n) {
          const int ks = kc % C::STAGES, vs = vc % C::STAGES;
          if (!__all_sync(FULL, mbar_wait(kv_full(ks), (kc / C::STAGES) & 1, abort_flag, lim) &&
                                    mbar_wait(kv_full(vs), (vc / C::STAGES) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s_tm = tbase + C::T_S + 128u * (j & 1);
          if (leader) {
            // S_j = Q K_j^T into buffer j&1 (issued after dQ(j-2), which read dS(j-2)
            // from the same columns)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t o = u16((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32);
              mma_ss(s_tm, dq0 + o, dkv0 + u16(ks * C::TILE_BYTES) + o, id_sq, kk > 0 ? 1u : 0u);
            }
          }
          // dP_j overwrites dP_{j-1}: the dS warpgroups must have read it
          if (j > 0 && !__all_sync(FULL, mbar_wait(dp_free, (j - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            // dP_j = dO V_j^T
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t o = u16((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32);
              mma_ss(tbase + C::T_DP, ddo0 + o, dkv0 + u16(vs * C::TILE_BYTES) + o, id_sq, kk > 0 ? 1u : 0u);
            }
            mma_commit(s_full(j & 1));
            mma_commit(kv_empty(vs));  // V_j is read only by dP_j
          }
        }
        if (j > 0) {
          const int i = j - 1, ks = (2 * i) % C::STAGES;
          if (!__all_sync(FULL, mbar_wait(ds_ready(i & 1), (i >> 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            // dQ += dS_i K_i: dS from TMEM (16-bit pairs over S_i's buffer: keys 0-63 at
            // columns 0-31, keys 64-127 at columns 64-95), K_i MN-major
            const uint32_t ds_tm = tbase + C::T_S + 128u * (i & 1);
            const uint64_t kd = dk_mn0 + u16(ks * C::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tbase + C::T_DQ, ds_tm + 64u * (kk / 4) + 8u * (kk % 4), kd + u16(kk * 2048), id_dq,
                     (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit(kv_empty(ks));
            if (i == n - 1) mma_commit(dq_done);
          }
        }
      }
      if (!ok && leader) fail();
      if (leader) mma_commit(final_bar);
      mbar_wait(final_bar, 0, nullptr, lim);
      // the last commits to kv_empty have no consumer: let them land before exit
      if (ok) {
        for (int c = (2 * n > C::STAGES ? 2 * n - C::STAGES : 0); c < 2 * n; ++c)
          mbar_wait(kv_empty(c % C::STAGES), (c / C::STAGES) & 1, nullptr, lim);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<200>();
    // ----------------------------------------------------------- dS warpgroups
    const int hf = warp >> 2;  // keys [64 hf, 64 hf + 64) of each block
    const int r = (warp & 3) * 32 + lane;
    const int row = r0 + r;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float cl2 = p.scale_log2;
    // -lse * log2(e) and -D of this query row, from the preprocess (-inf and 0 past N)
    const long long vrow = static_cast<long long>(bh) * p.Npad + row;
    const float nl2 = row < p.Npad ? p.l2vec[vrow] : -INFINITY;
    const float nd = row < p.Npad ? p.dvec[vrow] : 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(FULL, mbar_wait(s_full(j & 1), (j >> 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_tm = tbase + lane_off + C::T_S + 128u * (j & 1);
      const uint32_t dp_tm = tbase + lane_off + C::T_DP;
      const int nvis = CAUSAL && j == n - 1 ? row + 1 - 128 * j : 128;  // diagonal block
      {
        uint32_t sv[64], dpv[64];
        tmem_ld32(s_tm + 64u * hf, sv);
        tmem_ld32(s_tm + 64u * hf + 32u, sv + 32);
        tmem_ld32(dp_tm + 64u * hf, dpv);
        tmem_ld32(dp_tm + 64u * hf + 32u, dpv + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(dp_free);  // this warpgroup's half of dP_j is in registers
        const uint64_t cl2x2 = f2pack(cl2, cl2), nl2x2 = f2pack(nl2, nl2), ndx2 = f2pack(nd, nd);
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int c = 64 * hf + 2 * u;
          float a0, a1;
          f2unpack(ffma2(f2pack(__uint_as_float(sv[2 * u]), __uint_as_float(sv[2 * u + 1])), cl2x2, nl2x2), a0, a1);
          float p0 = dq_ex2(a0), p1 = dq_ex2(a1);
          if (CAUSAL) {
            if (c >= nvis) p0 = 0.f;
            if (c + 1 >= nvis) p1 = 0.f;
          }
          float d0, d1;
          f2unpack(fmul2(f2pack(p0, p1),
                         fadd2(f2pack(__uint_as_float(dpv[2 * u]), __uint_as_float(dpv[2 * u + 1])), ndx2)),
                   d0, d1);
          pk[u] = dq_pack2<BF16>(d0, d1);
        }
        // dS of this half -> 32 packed columns at the start of the half's own S columns
        // (already read by this thread; the other warpgroup reads only its own half)
        tmem_st32(s_tm + 64u * hf, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_ready(j & 1));
    }
    if (ok && !mbar_wait(dq_done, 0, abort_flag, lim)) ok = false;
    if (!ok) {
      *wg_fail = 1;
      fail();
    }
    named_bar_sync_n(1, 256);
    if (*wg_fail == 0) {  // uniform across both warpgroups
      tc_fence_after();
      uint16_t* out = p.dq + ((static_cast<long long>(b) * N + row) * p.Hq + h) * D;
#pragma unroll
      for (int c = hf * (D / 64); c < (hf + 1) * (D / 64); ++c) {  // this warpgroup's half of d
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + C::T_DQ + 32u * c, v);  // all lanes (.sync.aligned)
        tmem_wait_ld();
        if (row >= N) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 o;
          o.x = dq_pack2<BF16>(__uint_as_float(v[8 * u + 0]) * p.scale, __uint_as_float(v[8 * u + 1]) * p.scale);
          o.y = dq_pack2<BF16>(__uint_as_float(v[8 * u + 2]) * p.scale, __uint_as_float(v[8 * u + 3]) * p.scale);
          o.z = dq_pack2<BF16>(__uint_as_float(v[8 * u + 4]) * p.scale, __uint_as_float(v[8 * u + 5]) * p.scale);
          o.w = dq_pack2<BF16>(__uint_as_float(v[8 * u + 6]) * p.scale, __uint_as_float(v[8 * u + 7]) * p.scale);
          *reinterpret_cast<uint4*>(out + 32 * c + 8 * u) = o;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL>
static cudaError_t launch_bwd_dq_t(const BwdParams& p, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = fa_bwd_dq_kernel<D, BF16, CAUSAL>;
  cudaError_t e = prepare_launch_once<fa_bwd_dq_kernel<D, BF16, CAUSAL>>(C::SMEM, 384, 128 * 80 + 256 * 200);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((p.N + 127) / 128) * p.B * p.Hq;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream) {
  const bool bf = dtype == FA_BF16;
  if (d == 128) {
    if (bf) return causal ? launch_bwd_dq_t<128, true, true>(p, stream) : launch_bwd_dq_t<128, true, false>(p, stream);
    return causal ? launch_bwd_dq_t<128, false, true>(p, stream) : launch_bwd_dq_t<128, false, false>(p, stream);
  }
  if (bf) return causal ? launch_bwd_dq_t<64, true, true>(p, stream) : launch_bwd_dq_t<64, true, false>(p, stream);
  return causal ? launch_bwd_dq_t<64, false, true>(p, stream) : launch_bwd_dq_t<64, false, false>(p, stream);
}

}  // namespace fa
