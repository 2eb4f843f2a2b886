// Decode-shaped forward with the key range split across CTAs (split-KV).
//
// A few new queries per sequence (Nq, the tokens being generated) attend to a long
// key/value cache.  The pages separate this decode regime from prefill
// ("FlashAttention-2: atención eficiente en GPU para contextos largos", section "Cómo
// documentar una diferencia técnica") and motivate splitting work along the sequence
// when batch and heads alone leave the GPU idle (section "Tres mejoras en la
// utilización de la GPU"); the method is still exact attention.
//
// GB300 form:
//  * one CTA per (batch, key/value head, key split); the G = Hq/Hkv query heads of the
//    group and the Nq queries are packed into the rows of one 128-row tile (row
//    r = i*G + g), loaded by a single TMA box, so every key/value block read from HBM
//    serves the whole group;
//  * the same tcgen05 pipeline as the prefill kernel for that one tile: a TMA warp
//    streams K_j / V_j through a ring, an MMA warp issues S = Q K^T and O += P V with P
//    read from tensor memory, and one softmax warpgroup keeps m and l per row;
//  * each split writes its normalised partial output and log-sum-exp (fp32), and a
//    combine kernel merges the splits: lse = ln sum_s e^{lse_s},
//    O = sum_s e^{lse_s - lse} O_s.  With one split the kernel writes O and lse itself;
//  * two CTAs per SM (256 threads, 256 TMEM columns and < 100 KB shared memory each),
//    so the two CTAs' K/V streams overlap each other's serial softmax / MMA chain
//    (the softmax warpgroup runs with 176 registers, the control warps with 80);
//    the pass is bound by the HBM bytes of the cache.  With at most 8 (batch, kv head)
//    units at d = 128 a deeper K/V ring at one CTA per SM is used instead (the rule
//    and its measurements are in fa_decode_policy.h).
#include "fa_decode_policy.h"
#include "fa_internal.h"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

template <int D, bool DEEP>
struct DecCfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;  // Q tile, or one K / V block of 128 keys
  static constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 bytes
  // K/V ring: one block (K and V) in flight at two CTAs per SM, two with the deep ring
  static constexpr int STAGES = (D == 128 && !DEEP) ? 2 : 4;
  static constexpr int THREADS = 256;             // softmax warpgroup + control warpgroup
  static constexpr int NBARS = 4 + 2 * STAGES + 1;
  static constexpr int SMEM = 1024 + (1 + STAGES) * TILE_BYTES + 8 * NBARS + 64;
  static constexpr uint32_t TMEM_COLS = 256;      // S (128) and O (D <= 128)
  static_assert((DEEP ? 1 : 2) * SMEM <= 232448, "CTAs per SM");
};

__device__ __forceinline__ float dec_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Writes the result of a row that sees no key (o = 0, lse = -inf), or of an empty
// split (partial o = 0, partial lse = -inf: weight 0 in the combine).
template <int D>
__device__ __forceinline__ void dec_write_empty_row(const DecParams& p, int b, int hkv, int s, int r) {
  if (p.S == 1) {
    const int i = r / p.G, h = hkv * p.G + r % p.G;
    uint16_t* orow = p.o + ((static_cast<long long>(b) * p.Nq + i) * p.Hq + h) * D;
    for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0u, 0u, 0u, 0u);
    p.lse[(static_cast<long long>(b) * p.Hq + h) * p.Nq + i] = -INFINITY;
  } else {
    const long long prow = (static_cast<long long>(b * p.Hkv + hkv) * p.S + s) * p.M + r;
    float4* orow = reinterpret_cast<float4*>(p.opart + prow * D);
    for (int c = 0; c < D / 4; ++c) orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    p.lpart[prow] = -INFINITY;
  }
}

template <int D, bool BF16, bool CAUSAL, bool DEEP>
__global__ void __launch_bounds__(256, 2) fa_decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D, DEEP>;
  extern __shared__ uint8_t smem_raw_dec[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_dec) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::STAGES * C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0, s_full = bar0 + 8u, p_full = bar0 + 16u, o_done = bar0 + 24u;
  auto kv_full = [&](int st) { return bar0 + 8u * (4 + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (4 + C::STAGES + st); };
  const uint32_t final_bar = bar0 + 8u * (4 + 2 * C::STAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The split combine (launched as a programmatic dependent when there are several
  // splits) may be scheduled once every CTA of this grid is running; it still waits for
  // the whole grid to finish before it reads a partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- work decode: CTA = (batch, kv head, split); splits of one (b, kv head) are
  // consecutive CTAs
  const int s = static_cast<int>(blockIdx.x % p.S);
  const int bh = static_cast<int>(blockIdx.x / p.S);
  const int hkv = bh % p.Hkv;
  const int b = bh / p.Hkv;
  const int len_k = p.seqlens_k[b];
  if (len_k < 0 || len_k > p.Nmax) {
    if (threadIdx.x == 0 && s == 0 && hkv == 0) atomicOr(p.err, kDevErrSeqlens);
    return;  // uniform, before any barrier
  }
  const int nkb = (len_k + 127) / 128;
  const int jb0 = s * p.cps;
  const int n = max(0, min(nkb, jb0 + p.cps) - jb0);  // key blocks of this split
  // query i (row r = i*G + g) sees key j iff j < len_k and, with the mask, j <= i + off
  const int off = len_k - p.Nq;
  const int lim0 = CAUSAL ? max(0, min(len_k, off + 1)) : len_k;  // keys seen by query 0
  const int nfull = lim0 / 128;  // blocks every row sees completely
  if (n == 0) {
    for (int r = threadIdx.x; r < p.M; r += blockDim.x) dec_write_empty_row<D>(p, b, hkv, s, r);
    return;
  }

  // rows [M, 128) of the query tile are not written by the copy: zero them so every
  // row the tensor core reads is finite
  if (p.M < 128) {
    for (int i = threadIdx.x; i < C::CHUNKS * (128 - p.M) * 8; i += blockDim.x) {
      const int ch = i / ((128 - p.M) * 8), rem = i % ((128 - p.M) * 8);
      *reinterpret_cast<uint4*>(sQ + ch * C::CHUNK_BYTES + (p.M + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *wg_fail = 0;
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
    }
    mbar_init(final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
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

  if (warp >= 4) {
    setmaxnreg_dec<80>();
    const bool leader = elect_one();
    if (warp == 4) {
      // ------------------------------------------------------------ TMA producer
      if (leader) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        // the group's query heads x the new queries: one box per 64-column chunk
        mbar_arrive_expect_tx(q_full, C::CHUNKS * p.M * 128);
        for (int ch = 0; ch < C::CHUNKS; ++ch)
          tma_load_4d(smem_u32(sQ + ch * C::CHUNK_BYTES), &p.tm_q, q_full, ch * 64, hkv * p.G, 0, b);
      }
      int c = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind, ++c) {
          const int slot = c % C::STAGES;
          if (c >= C::STAGES &&
              !__all_sync(FULL, mbar_wait(kv_empty(slot), ((c / C::STAGES) - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(kv_full(slot), C::TILE_BYTES);
            const CUtensorMap* map = kind ? &p.tm_v : &p.tm_k;
            // contiguous cache: rows 128 (jb0 + j) of sequence b; paged cache: all 128 rows
            // of the block's page (a page index outside the cache reads zeros and is
            // reported)
            int row = 128 * (jb0 + j), outer = b;
            if (p.block_table != nullptr) {
              outer = p.block_table[static_cast<long long>(b) * p.max_pages + jb0 + j];
              row = 0;
              if (kind == 0 && (outer < 0 || outer >= p.num_pages)) atomicOr(p.err, kDevErrSeqlens);
            }
            for (int ch = 0; ch < C::CHUNKS; ++ch)
              tma_load_4d(smem_u32(sKV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES), map, kv_full(slot), ch * 64,
                          hkv, row, outer);
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
    } else if (warp == 5) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t id_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t id_pv = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
      bool ok = __all_sync(FULL, mbar_wait(q_full, 0, abort_flag, lim));
      const uint32_t s_tm = tbase, o_tm = tbase + 128u;
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dkv0 = smem_desc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sKV), C::CHUNK_BYTES, 1024);
      for (int j = 0; j <= n && ok; ++j) {
        const int kc = 2 * j, vc = 2 * j - 1;
        const int kslot = kc % C::STAGES, vslot = (vc + C::STAGES) % C::STAGES;
        if (j < n && !__all_sync(FULL, mbar_wait(kv_full(kslot), (kc / C::STAGES) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        if (j > 0) {
          if (!__all_sync(FULL, mbar_wait(kv_full(vslot), (vc / C::STAGES) & 1, abort_flag, lim) &&
                                    mbar_wait(p_full, (j - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O += P(j-1) V_{j-1}: P from TMEM over S's columns, V MN-major
          const uint64_t vd = dv0 + static_cast<uint64_t>((vslot * C::TILE_BYTES) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(o_tm, s_tm + 8u * kk, vd + static_cast<uint64_t>((kk * 2048) >> 4), id_pv,
                     (j - 1 > 0 || kk > 0) ? 1u : 0u);
            if (j == n) mma_commit(o_done);
          }
        }
        tc_fence_after();
        if (j < n) {
          // S = Q K_j^T (in issue order after the product above, which read P from the
          // same columns)
          const uint64_t kd = dkv0 + static_cast<uint64_t>((kslot * C::TILE_BYTES) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t o16 = static_cast<uint64_t>(((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32) >> 4);
              mma_ss(s_tm, dq0 + o16, kd + o16, id_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(s_full);
          }
        }
        if (leader) {
          if (j > 0) mma_commit(kv_empty(vslot));
          if (j < n) mma_commit(kv_empty(kslot));
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
    setmaxnreg_inc<176>();
    // ------------------------------------------------------------ softmax warpgroup
    const int r = warp * 32 + lane;  // packed row = TMEM lane
    const int i = min(r / p.G, p.Nq - 1);  // query (rows past M are padding)
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const uint32_t s_tm = tbase + lane_off, o_tm = tbase + lane_off + 128u;
    const float cl2 = p.scale_log2;
    const int lim_row = CAUSAL ? min(len_k, i + off + 1) : len_k;  // keys [0, lim_row) visible
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(FULL, mbar_wait(s_full, j & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp * 32 >= p.M) {
        // every row of this warp is padding: keep the barrier protocol, skip the work
        // (its P stays whatever S left there; padding rows' outputs are never stored)
        tc_fence_before();
        mbar_arrive(p_full);
        continue;
      }
      // Two passes over S in 64-column halves (the row maximum first, then the
      // exponentials), so a thread holds 64 scores instead of 128 and the softmax
      // warpgroup fits the 176 registers two CTAs per SM leave it.
      const int jg = jb0 + j;
      const bool masked = jg >= nfull;
      const int nvis = lim_row - 128 * jg;  // columns [0, nvis) of this block are visible
      float mx = -INFINITY;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[64];
        tmem_ld32(s_tm + 64u * hf, sr);
        tmem_ld32(s_tm + 64u * hf + 32u, sr + 32);
        tmem_wait_ld();
        float* v = reinterpret_cast<float*>(sr);
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (64 * hf + c >= nvis) v[c] = -INFINITY;
        }
        // four independent chains of three-input maxima
        float m0 = fmax3(mx, v[0], v[1]), m1 = fmax3(v[2], v[3], v[4]), m2 = fmax3(v[5], v[6], v[7]);
        float m3 = fmax3(v[8], v[9], v[10]);
#pragma unroll
        for (int c = 11; c + 8 <= 59; c += 8) {
          m0 = fmax3(m0, v[c], v[c + 1]);
          m1 = fmax3(m1, v[c + 2], v[c + 3]);
          m2 = fmax3(m2, v[c + 4], v[c + 5]);
          m3 = fmax3(m3, v[c + 6], v[c + 7]);
        }
        m0 = fmax3(m0, v[59], v[60]);
        m1 = fmax3(m1, v[61], v[62]);
        mx = fmax3(fmax3(m0, m1, m2), m3, v[63]);
      }
      if (j == 0) {
        m = mx;
      } else if (__any_sync(FULL, (mx - m) * cl2 > 8.0f)) {
        // lazy correction (PV(j-1) is complete: S(j) was issued after it)
        const float m_new = fmaxf(m, mx);
        const float alpha = (m_new == -INFINITY) ? 1.f : dec_ex2((m - m_new) * cl2);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(o_tm + 32u * c, orr);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) orr[u] = __float_as_uint(__uint_as_float(orr[u]) * alpha);
          tmem_st32(o_tm + 32u * c, orr);
        }
        tmem_wait_st();
      }
      // a row with no visible key so far keeps m = -inf and gets p = 0
      const float neg = (m == -INFINITY) ? 0.f : -m * cl2;
      const uint64_t cl2x2 = f2pack(cl2, cl2), negx2 = f2pack(neg, neg);
      float sum = 0.f;
      // P of half hf goes to packed columns [32 hf, 32 hf + 32), over S columns this
      // thread has already read (half 1's scores, columns 64-127, are untouched by it)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[64];
        tmem_ld32(s_tm + 64u * hf, sr);
        tmem_ld32(s_tm + 64u * hf + 32u, sr + 32);
        tmem_wait_ld();
        uint32_t pk[32];
        uint64_t acc = 0ull;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int c = 64 * hf + 2 * u;
          const float s0 = (masked && c >= nvis) ? -INFINITY : __uint_as_float(sr[2 * u]);
          const float s1 = (masked && c + 1 >= nvis) ? -INFINITY : __uint_as_float(sr[2 * u + 1]);
          float a0, a1;
          f2unpack(ffma2(f2pack(s0, s1), cl2x2, negx2), a0, a1);
          const float p0 = dec_ex2(a0), p1 = dec_ex2(a1);
          acc = fadd2(acc, f2pack(p0, p1));
          pk[u] = pack_half2<BF16>(p0, p1);
        }
        float sa, sb;
        f2unpack(acc, sa, sb);
        sum += sa + sb;
        tmem_st32(s_tm + 32u * hf, pk);
      }
      l += sum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && !mbar_wait(o_done, 0, abort_flag, lim)) ok = false;
    if (!ok) {
      *wg_fail = 1;
      fail();
    }
    named_bar_sync_n(1, 128);
    if (*wg_fail == 0) {
      tc_fence_after();
      const bool has = l > 0.f;
      const float inv = has ? 1.0f / l : 0.f;
      const float lse = has ? m * p.scale + logf(l) : -INFINITY;
      const bool live = r < p.M;
      const int h = hkv * p.G + r % p.G;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(o_tm + 32u * c, orr);
        tmem_wait_ld();
        if (!live) continue;
        if (p.S == 1) {
          uint16_t* orow = p.o + ((static_cast<long long>(b) * p.Nq + i) * p.Hq + h) * D + 32 * c;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_half2<BF16>(__uint_as_float(orr[8 * u + 0]) * inv, __uint_as_float(orr[8 * u + 1]) * inv);
            w.y = pack_half2<BF16>(__uint_as_float(orr[8 * u + 2]) * inv, __uint_as_float(orr[8 * u + 3]) * inv);
            w.z = pack_half2<BF16>(__uint_as_float(orr[8 * u + 4]) * inv, __uint_as_float(orr[8 * u + 5]) * inv);
            w.w = pack_half2<BF16>(__uint_as_float(orr[8 * u + 6]) * inv, __uint_as_float(orr[8 * u + 7]) * inv);
            reinterpret_cast<uint4*>(orow)[u] = w;
          }
        } else {
          const long long prow = (static_cast<long long>(bh) * p.S + s) * p.M + r;
          float4* orow = reinterpret_cast<float4*>(p.opart + prow * D + 32 * c);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            orow[u] = make_float4(__uint_as_float(orr[4 * u]) * inv, __uint_as_float(orr[4 * u + 1]) * inv,
                                  __uint_as_float(orr[4 * u + 2]) * inv, __uint_as_float(orr[4 * u + 3]) * inv);
        }
      }
      if (live) {
        if (p.S == 1)
          p.lse[(static_cast<long long>(b) * p.Hq + h) * p.Nq + i] = lse;
        else
          p.lpart[(static_cast<long long>(bh) * p.S + s) * p.M + r] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// Merges the splits of every packed row: lse = ln sum_s e^{lse_s},
// O = sum_s e^{lse_s - lse} O_s (a split that saw no key has lse_s = -inf, weight 0).
// Four warps share a row (two rows per CTA): each takes the row's lse from all splits
// (lanes over splits, a running maximum and rescaled sum per lane, then combined across
// the warp), adds the partial rows of its own splits s = q, q + 4, ... (lane owns D/32
// columns; eight row loads in flight), and the four sums meet in shared memory.  With
// few rows this spreads a row's reads over four warps.  Launched as a programmatic
// dependent of fa_decode_kernel: griddepcontrol.wait returns once that grid has
// finished and its writes are visible, so the launch itself overlaps its tail.
constexpr int kCombWarpsPerRow = 4;

template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_decode_combine(const __grid_constant__ DecParams p) {
  constexpr int V = D / 32;  // columns per lane: 4 (d = 128) or 2 (d = 64)
  constexpr int WPR = kCombWarpsPerRow, RPC = 8 / WPR;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ float red[8][D];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp % WPR, slot = warp / WPR;
  const long long rows = static_cast<long long>(p.B) * p.Hkv * p.M;
  const int nmine = (p.S - q + WPR - 1) / WPR;  // splits q, q + WPR, ... of this warp
  for (long long r0 = static_cast<long long>(blockIdx.x) * RPC; r0 < rows;
       r0 += static_cast<long long>(gridDim.x) * RPC) {  // uniform over the CTA
    const long long w = r0 + slot;
    const bool valid = w < rows;
    float acc[V];
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = 0.f;
    float lse = -INFINITY;
    int r = 0, hkv = 0, b = 0;
    if (valid) {  // uniform over the warp
      r = static_cast<int>(w % p.M);
      const long long bh = w / p.M;
      hkv = static_cast<int>(bh % p.Hkv);
      b = static_cast<int>(bh / p.Hkv);
      const long long base = bh * p.S * p.M + r;  // partial row of split s: base + s*M
      const float* lp = p.lpart + base;
      float m = -INFINITY, t = 0.f;
      for (int s = lane; s < p.S; s += 32) {
        const float x = lp[static_cast<long long>(s) * p.M];
        if (x > m) {
          t = t * expf(m - x) + 1.f;  // e^{-inf} = 0 on the first finite value
          m = x;
        } else if (x != -INFINITY) {
          t += expf(x - m);
        }
      }
      float mx = m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
      if (mx != -INFINITY) {
        float tot = m == -INFINITY ? 0.f : t * expf(m - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
        lse = mx + logf(tot);
        const float* op = p.opart + base * D + lane * V;
        for (int c0 = 0; c0 < nmine; c0 += 32) {
          const int mine = c0 + lane;
          const float wl =
              mine < nmine ? expf(lp[static_cast<long long>(q + WPR * mine) * p.M] - lse) : 0.f;
          const int n = min(32, nmine - c0);
          for (int j0 = 0; j0 < n; j0 += 8) {
            float v[8][V];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (j0 + u < n) {
                const float* src = op + static_cast<long long>(q + WPR * (c0 + j0 + u)) * p.M * D;
                if constexpr (V == 4) {
                  const float4 x4 = *reinterpret_cast<const float4*>(src);
                  v[u][0] = x4.x, v[u][1] = x4.y, v[u][2] = x4.z, v[u][3] = x4.w;
                } else {
                  const float2 x2 = *reinterpret_cast<const float2*>(src);
                  v[u][0] = x2.x, v[u][1] = x2.y;
                }
              } else {
#pragma unroll
                for (int c = 0; c < V; ++c) v[u][c] = 0.f;
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float wj = __shfl_sync(FULL, wl, (j0 + u) & 31);
              if (j0 + u < n && wj > 0.f) {
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = fmaf(wj, v[u][c], acc[c]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < V; ++c) red[warp][lane * V + c] = acc[c];
    __syncthreads();
    if (valid && q == 0) {
#pragma unroll
      for (int k = 1; k < WPR; ++k)
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] += red[warp + k][lane * V + c];
      const int i = r / p.G, h = hkv * p.G + r % p.G;
      uint16_t* orow = p.o + ((static_cast<long long>(b) * p.Nq + i) * p.Hq + h) * D + lane * V;
      if constexpr (V == 4) {
        uint2 o2;
        o2.x = pack_half2<BF16>(acc[0], acc[1]);
        o2.y = pack_half2<BF16>(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(orow) = o2;
      } else {
        *reinterpret_cast<uint32_t*>(orow) = pack_half2<BF16>(acc[0], acc[1]);
      }
      if (lane == 0) p.lse[(static_cast<long long>(b) * p.Hq + h) * p.Nq + i] = lse;
    }
    __syncthreads();
  }
}

template <int D, bool BF16, bool CAUSAL, bool DEEP = false>
static cudaError_t launch_decode_t(const DecParams& p, cudaStream_t stream) {
  using C = DecCfg<D, DEEP>;
  auto kern = fa_decode_kernel<D, BF16, CAUSAL, DEEP>;
  cudaError_t e = prepare_launch_once<fa_decode_kernel<D, BF16, CAUSAL, DEEP>>(C::SMEM, 256, 128 * 80 + 128 * 176);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.B) * p.Hkv * p.S;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.S == 1) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hkv * p.M;
  const long long blocks = (rows + 8 / kCombWarpsPerRow - 1) / (8 / kCombWarpsPerRow);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks < 4096 ? blocks : 4096));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_decode_combine<D, BF16>, p);
}

cudaError_t launch_decode(const DecParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream) {
  const bool bf = dtype == FA_BF16;
  if (d == 128 && decode_deep_ring(d, static_cast<long long>(p.B) * p.Hkv)) {
    if (bf)
      return causal ? launch_decode_t<128, true, true, true>(p, stream) : launch_decode_t<128, true, false, true>(p, stream);
    return causal ? launch_decode_t<128, false, true, true>(p, stream) : launch_decode_t<128, false, false, true>(p, stream);
  }
  if (d == 128) {
    if (bf) return causal ? launch_decode_t<128, true, true>(p, stream) : launch_decode_t<128, true, false>(p, stream);
    return causal ? launch_decode_t<128, false, true>(p, stream) : launch_decode_t<128, false, false>(p, stream);
  }
  if (bf) return causal ? launch_decode_t<64, true, true>(p, stream) : launch_decode_t<64, true, false>(p, stream);
  return causal ? launch_decode_t<64, false, true>(p, stream) : launch_decode_t<64, false, false>(p, stream);
}

}  // namespace fa
