// Forward pass of exact attention on sm_103a: O = softmax(scale * Q K^T [+ causal]) V.
//
// Method ("FlashAttention-2: atención eficiente en GPU para contextos largos",
// sections "Bloques pequeños, normalización global" and "Tres mejoras en la
// utilización de la GPU"): key/value blocks stream through on-chip memory while a
// running row maximum m and row sum l are kept per query row; partial outputs are
// rescaled when m grows, so the final O / l is the globally normalised result and
// the N x N score / probability matrices never reach device memory.
//
// GB300 form of that design:
//  * one CTA owns 2 query tiles of 128 rows of one (batch, head); work is split
//    along the sequence as well as batch and heads;
//  * a TMA warp streams Q once and K_j / V_j through a ring of shared-memory stages
//    (128-byte swizzle, mbarrier transaction counts);
//  * an MMA warp issues tcgen05.mma: S_t = Q_t K_j^T into tensor memory (TMEM), and
//    O_t += P_t V_j with P_t read straight from TMEM, where the softmax left it;
//  * one softmax warpgroup per query tile (thread = row = TMEM lane) reads S_t,
//    applies the mask only on the block that needs it (diagonal block for causal,
//    last block when N is not a multiple of 128), keeps m and l in registers with
//    the scale folded into the exp2 argument, writes P_t as 16-bit pairs over S_t,
//    and rescales O_t in TMEM only when the running maximum grew by more than
//    2^8 (the result is exact for any threshold, since O and l carry the same
//    factor);
//  * the epilogue divides by l, rounds to 16 bits, stages the tile in shared memory
//    and TMA-stores it (rows >= N are clipped by the tensor map), and writes
//    lse = scale * m + ln(l).
#include "fa_internal.h"
#include "fa_math.cuh"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                  // query rows per tile (one TMEM lane each)
  static constexpr int BN = 128;                  // keys per block
  static constexpr int TILES = 2;                 // query tiles per CTA
  static constexpr int CHUNKS = D / 64;           // 128-byte swizzle column chunks of a row
  static constexpr int TILE_BYTES = 128 * D * 2;  // one Q, K or V tile
  static constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  static constexpr int THREADS = 384;             // 2 softmax warpgroups + control warpgroup
  // registers after setmaxnreg: control warpgroup 80, softmax warpgroups 208 each; the
  // total must fit the launch allocation of 384 x 168 = 64512 (checked before launch)
  static constexpr int REG_CTRL = 80, REG_SOFTMAX = 208;
  static constexpr int REG_SPLIT = 128 * REG_CTRL + 256 * REG_SOFTMAX;
  static_assert(REG_SPLIT <= 384 * 168, "register split above the launch allocation");
  static constexpr int NBARS = 8 + 2 * STAGES + 1;
  static constexpr int SMEM = 1024 + TILES * TILE_BYTES + STAGES * TILE_BYTES + 8 * NBARS + 64;
  static constexpr uint32_t TMEM_COLS = 512;      // S_0, S_1 (128 each), O_0, O_1 (D each)
  static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float ex2f(float x) { return ex2_mufu(x); }

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(384, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILES * C::TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::STAGES * C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]

  const uint32_t bar0 = smem_u32(bars);
  auto q_full = [&](int t) { return bar0 + 8u * (0 + t); };
  auto s_full = [&](int t) { return bar0 + 8u * (2 + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (4 + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (6 + t); };
  auto kv_full = [&](int s) { return bar0 + 8u * (8 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (8 + C::STAGES + s); };
  const uint32_t final_bar = bar0 + 8u * (8 + 2 * C::STAGES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work decode.  Without the mask every tile costs the same, and the query
  // blocks of one (batch, head) are consecutive CTAs so the resident CTAs share a few
  // heads' K/V through L2.  With the causal mask tiles are issued heaviest first
  // (largest query offset) across all heads, which balances the last waves.
  // Consecutive heads of a GQA group share K/V in both orders.
  const int N = VARLEN ? p.vl.max_q : p.N;  // query rows the grid covers per sequence
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
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  // Sequence geometry.  Fixed length: len_q = len_k = N.  Variable length: sequence b
  // sits at rows [start, start + len) of the packed tensors, and with the causal mask
  // query i sees key j iff j <= i + (len_k - len_q) (the mask is aligned at the
  // bottom-right corner, so the last query sees every key).
  int start_q = 0, len_q = N, start_k = 0, len_k = N;
  if (VARLEN) {
    if (!seq_span(p.vl, b, start_q, len_q, start_k, len_k)) {
      if (threadIdx.x == 0 && qb == 0) atomicOr(p.err, kDevErrSeqlens);
      return;  // uniform, before any barrier or TMEM allocation
    }
    if (qb * 256 >= len_q) return;
  }
  const int off = len_k - len_q;
  // query tile t covers rows [qb*256 + 128t, +128) and visits n_t key blocks; with
  // variable length the first nf_t of them need no mask for any row of the tile
  const int r00 = qb * 256, r01 = qb * 256 + 128;
  auto nblocks = [&](int r0) {
    if (r0 >= len_q) return 0;
    if (!VARLEN) return CAUSAL ? r0 / 128 + 1 : (N + 127) / 128;
    const int ve = CAUSAL ? min(len_k, r0 + 128 + off) : len_k;  // keys seen by the tile's last row
    return ve > 0 ? (ve + 127) / 128 : 0;
  };
  auto nfull = [&](int r0) { return max(0, CAUSAL ? min(len_k, r0 + off + 1) : len_k) / 128; };
  const int n0 = nblocks(r00), n1 = nblocks(r01);
  auto n_of = [&](int t) { return t ? n1 : n0; };
  auto r0_of = [&](int t) { return t ? r01 : r00; };
  const int nmax = n0 > n1 ? n0 : n1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    wg_fail[0] = wg_fail[1] = 0;
    for (int i = 0; i < 8; ++i) mbar_init(bar0 + 8u * i, (i >= 4 && i < 6) ? 128u : 1u);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(final_bar, 1);
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
  const volatile int* no_abort = nullptr;  // waits that must not give up early on abort

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.err, kDevErrTimeout);
  };

  if (warp >= 8) {
   // control warpgroup gives registers to the softmax warpgroups (C::REG_SPLIT)
   setmaxnreg_dec<C::REG_CTRL>();
   // The control warps run their loops with all 32 lanes (warp-uniform control flow,
   // so loop state and descriptors live in uniform registers); one elected lane issues
   // the TMA copies, the tcgen05 instructions and their commits.
   constexpr unsigned FULL = 0xffffffffu;
   const bool leader = elect_one();
   if (warp == 8) {
    // ------------------------------------------------------------- TMA producer
    if (leader) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      for (int t = 0; t < 2; ++t) {
        if (n_of(t) == 0) continue;
        mbar_arrive_expect_tx(q_full(t), C::TILE_BYTES);
        for (int ch = 0; ch < C::CHUNKS; ++ch) {
          const uint32_t dst = smem_u32(sQ + t * C::TILE_BYTES + ch * C::CHUNK_BYTES);
          if (VARLEN)
            tma_load_3d(dst, &p.tm_q, q_full(t), ch * 64, h, start_q + r0_of(t));
          else
            tma_load_4d(dst, &p.tm_q, q_full(t), ch * 64, h, r0_of(t), b);
        }
      }
    }
    int c = 0;
    bool ok = true;
    for (int j = 0; j < nmax && ok; ++j) {
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
          for (int ch = 0; ch < C::CHUNKS; ++ch) {
            const uint32_t dst = smem_u32(sKV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES);
            if (VARLEN)
              tma_load_3d(dst, map, kv_full(slot), ch * 64, hkv, start_k + 128 * j);
            else
              tma_load_4d(dst, map, kv_full(slot), ch * 64, hkv, 128 * j, b);
          }
        }
      }
    }
    if (!ok) {
      if (leader) fail();
      // let copies already in flight land before the CTA's shared memory goes away
      for (int i = (c > C::STAGES ? c - C::STAGES : 0); i < c; ++i)
        mbar_wait(kv_full(i % C::STAGES), (i / C::STAGES) & 1, no_abort, lim);
      for (int t = 0; t < 2; ++t)
        if (n_of(t)) mbar_wait(q_full(t), 0, no_abort, lim);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_qk = idesc_f16(128, 128, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t id_pv = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
    bool ok = true;
    for (int t = 0; t < 2 && ok; ++t)
      if (n_of(t)) ok = __all_sync(FULL, mbar_wait(q_full(t), 0, abort_flag, lim));
    const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
    // descriptor templates; per k-step only the start-address field (bits 0-13, in
    // 16-byte units) moves, and it never carries out of its field inside the CTA's
    // shared memory window
    const uint64_t dq0 = smem_desc_sw128(sq, 16, 1024), dkv0 = smem_desc_sw128(skv, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(skv, C::CHUNK_BYTES, 1024);
    for (int j = 0; j <= nmax && ok; ++j) {
      const int kc = 2 * j, vc = 2 * j - 1;
      const int kslot = kc % C::STAGES, vslot = (vc + C::STAGES) % C::STAGES;
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
        const uint32_t s_tm = tbase + 128u * t;
        const uint32_t o_tm = tbase + 256u + uint32_t(D) * t;
        if (j > 0 && j - 1 < n_of(t)) {
          // O_t += P_t(j-1) V_{j-1}: P_t from TMEM (16-bit pairs over S_t), V MN-major.
          if (!__all_sync(FULL, mbar_wait(p_full(t), (j - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // MN-major operand: leading-dimension offset = stride between 64-column
          // chunks, stride-dimension offset = stride between 8-key row groups.
          const uint64_t vd = dv0 + static_cast<uint64_t>((vslot * C::TILE_BYTES) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(o_tm, s_tm + 8u * kk, vd + static_cast<uint64_t>((kk * 2048) >> 4), id_pv,
                     (j - 1 > 0 || kk > 0) ? 1u : 0u);
            if (j - 1 == n_of(t) - 1) mma_commit(o_done(t));
          }
        }
        if (j < n_of(t)) {
          // S_t = Q_t K_j^T, both K-major.
          const uint64_t qd = dq0 + static_cast<uint64_t>((t * C::TILE_BYTES) >> 4);
          const uint64_t kd = dkv0 + static_cast<uint64_t>((kslot * C::TILE_BYTES) >> 4);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = static_cast<uint64_t>(((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32) >> 4);
              mma_ss(s_tm, qd + off, kd + off, id_qk, kk > 0 ? 1u : 0u);
            }
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
    // every MMA the leader issued must be finished before TMEM is released
    if (leader) mma_commit(final_bar);
    mbar_wait(final_bar, 0, no_abort, lim);
    // The last commits to kv_empty have no consumer; let their arrivals land before this
    // CTA's shared memory (and the barriers in it) passes to the next CTA.
    if (ok) {
      for (int c = (2 * nmax > C::STAGES ? 2 * nmax - C::STAGES : 0); c < 2 * nmax; ++c)
        mbar_wait(kv_empty(c % C::STAGES), (c / C::STAGES) & 1, no_abort, lim);
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<C::REG_SOFTMAX>();
    // ----------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;
    const int rit = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t s_tm = tbase + lane_off + 128u * t;
    const uint32_t o_tm = tbase + lane_off + 256u + uint32_t(D) * t;
    const float cl2 = p.scale_log2;
    const int row = r0_of(t) + rit;
    const int nf = nfull(r0_of(t));
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_of(t); ++j) {
      // warp-uniform outcome: the tcgen05.ld / vote below need all 32 lanes
      if (!__all_sync(0xffffffffu, mbar_wait(s_full(t), j & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + 32u * c, sr + 32 * c);
      tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sr);
      if (VARLEN ? j >= nf : (j == n_of(t) - 1 && (CAUSAL || (N & 127)))) {
        // keys k0 + c are visible for c < nvis (key < len_k, and key <= row + off with
        // the mask)
        const int k0 = 128 * j;
        const int nvis = CAUSAL ? min(len_k, row + off + 1) - k0 : len_k - k0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= nvis) s[c] = -INFINITY;
      }
      const float mx = rowmax128(s);
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, (mx - m) * cl2 > 8.0f)) {
        // lazy correction: bring O and l to the new maximum (needs PV_t(j-1) done,
        // which the completion of S_t(j), issued after it, already implies)
        const float m_new = fmaxf(m, mx);
        // (a row that sees no key keeps m = -inf; its O and l stay 0)
        const float alpha = (VARLEN && CAUSAL && m_new == -INFINITY) ? 1.f : ex2f((m - m_new) * cl2);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(o_tm + 32u * c, orr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(o_tm + 32u * c, orr);
        }
        tmem_wait_st();
      }
      // a row with no visible key so far (only possible with variable lengths and the
      // mask) has m = -inf: its p are exp2(-inf) = 0
      const float neg = (VARLEN && CAUSAL && m == -INFINITY) ? 0.f : -m * cl2;
      // exponent arguments two at a time (f32x2 FMA), sums in two packed accumulators
      const uint64_t cl2x2 = f2pack(cl2, cl2), negx2 = f2pack(neg, neg);
      uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        float a0, a1, a2, a3;
        f2unpack(ffma2(f2pack(s[c], s[c + 1]), cl2x2, negx2), a0, a1);
        f2unpack(ffma2(f2pack(s[c + 2], s[c + 3]), cl2x2, negx2), a2, a3);
        s[c] = ex2f(a0);
        s[c + 1] = ex2f(a1);
        s[c + 2] = ex2f(a2);
        s[c + 3] = ex2f(a3);
        acc0 = fadd2(acc0, f2pack(s[c], s[c + 1]));
        acc1 = fadd2(acc1, f2pack(s[c + 2], s[c + 3]));
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
      mbar_arrive(p_full(t));
    }
    if (n_of(t) > 0) {
      if (ok && !mbar_wait(o_done(t), 0, abort_flag, lim)) ok = false;
      if (!ok) {
        wg_fail[t] = 1;
        fail();
      }
      // every thread of the warpgroup reaches this barrier; afterwards wg_fail[t]
      // is read-only, so the branch below is uniform across the warpgroup
      named_bar_sync_n(1 + t, 128);
      if (wg_fail[t] == 0) {
        tc_fence_after();
        // ---- epilogue: O / l -> 16-bit -> swizzled staging (Q_t's buffer) -> TMA store.
        // A variable-length tile that ends past its sequence is written row by row
        // instead (a tile store would run into the next sequence's rows).
        const float inv = (VARLEN && CAUSAL) ? (l > 0.f ? 1.0f / l : 0.f) : 1.0f / l;
        const bool direct = VARLEN && r0_of(t) + 128 > len_q;
        uint16_t* orow = p.o + (static_cast<long long>(start_q + row) * p.Hq + h) * D;
        uint8_t* stage = sQ + t * C::TILE_BYTES;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(o_tm + 32u * c, orr);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_half2<BF16>(__uint_as_float(orr[2 * i]) * inv, __uint_as_float(orr[2 * i + 1]) * inv);
          if (direct) {
            if (row < len_q) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(orow + 32 * c + 8 * u) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            continue;
          }
          uint8_t* rowp = stage + (c >> 1) * C::CHUNK_BYTES + rit * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = (c & 1) * 4 + u;
            const int phys = unit ^ (rit & 7);
            *reinterpret_cast<uint4*>(rowp + phys * 16) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        if (!direct) {  // uniform across the warpgroup
          fence_proxy_async_smem();
          named_bar_sync_n(3 + t, 128);
          if (rit == 0) {
            for (int ch = 0; ch < C::CHUNKS; ++ch) {
              if (VARLEN)
                tma_store_3d(&p.tm_o, smem_u32(stage + ch * C::CHUNK_BYTES), ch * 64, h, start_q + r0_of(t));
              else
                tma_store_4d(&p.tm_o, smem_u32(stage + ch * C::CHUNK_BYTES), ch * 64, h, r0_of(t), b);
            }
            bulk_commit_group();
            // the staging (Q_t's buffer) must outlive the copy's reads of it; the global
            // writes need no wait (they complete before the kernel does)
            bulk_wait_group_read0();
          }
        }
        if (row < len_q) {
          const float lse = (VARLEN && CAUSAL && !(l > 0.f)) ? -INFINITY : m * p.scale + logf(l);
          if (VARLEN)
            p.lse[static_cast<size_t>(h) * p.vl.total_q + start_q + row] = lse;
          else
            p.lse[(static_cast<size_t>(b) * p.Hq + h) * N + row] = lse;
        }
      }
    } else if (VARLEN && r0_of(t) < len_q) {
      // no key is visible to any row of this tile: O = 0 and lse = ln 0 = -inf
      if (row < len_q) {
        uint16_t* orow = p.o + (static_cast<long long>(start_q + row) * p.Hq + h) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) *reinterpret_cast<uint4*>(orow + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
        p.lse[static_cast<size_t>(h) * p.vl.total_q + start_q + row] = -INFINITY;
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

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
static cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL, VARLEN>;
  cudaError_t e = prepare_launch_once<fa_fwd_kernel<D, BF16, CAUSAL, VARLEN>>(C::SMEM, C::THREADS, C::REG_SPLIT);
  if (e != cudaSuccess) return e;
  const long long nqb = ((VARLEN ? p.vl.max_q : p.N) + 255) / 256;
  const long long grid = nqb * p.B * p.Hq;
  kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_fwd_d(const FwdParams& p, bool causal, bool varlen, cudaStream_t stream) {
  if (varlen) return causal ? launch_fwd_t<D, BF16, true, true>(p, stream) : launch_fwd_t<D, BF16, false, true>(p, stream);
  return causal ? launch_fwd_t<D, BF16, true, false>(p, stream) : launch_fwd_t<D, BF16, false, false>(p, stream);
}

cudaError_t launch_fwd(const FwdParams& p, int d, fa_dtype dtype, bool causal, bool varlen, cudaStream_t stream) {
  const bool bf = dtype == FA_BF16;
  if (d == 128) return bf ? launch_fwd_d<128, true>(p, causal, varlen, stream) : launch_fwd_d<128, false>(p, causal, varlen, stream);
  return bf ? launch_fwd_d<64, true>(p, causal, varlen, stream) : launch_fwd_d<64, false>(p, causal, varlen, stream);
}

}  // namespace fa
