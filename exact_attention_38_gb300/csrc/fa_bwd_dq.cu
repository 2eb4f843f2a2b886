// dQ of the backward pass in a fixed summation order (the deterministic backward).
//
// The main backward kernel owns a block of keys and adds its dS K contribution into an
// fp32 dQ accumulator with tensor-memory-access reductions; the order in which CTAs
// land their additions varies from run to run, so dQ's last bits do too.  This kernel
// instead owns 256 queries (two tiles of 128) and walks the key blocks in ascending order,
// recomputing S = Q K^T and dP = dO V^T and accumulating dQ = scale * sum_j dS_j K_j in
// tensor memory: every dQ element is then summed in the same order on every run.  The
// price is two more GEMM-shaped products per (query, key) block (S and dP are computed
// by both kernels).  The gradient is the closed form of the pages' exact attention
// ("FlashAttention-2: atención eficiente en GPU para contextos largos", section "Bloques
// pequeños, normalización global"): dS = P * (dP - D), P = exp(s - lse).
//
// GB300 form (two 128-query tiles of one (batch, query head) per CTA, 384 threads):
//  * warp 8 loads Q and dO of both tiles once and streams K_j / V_j through a ring shared by
//    the two tiles (each K/V block read from L2 serves 256 queries);
//  * tile t owns a 128-column TMEM buffer used three times per key block: S_t = Q_t K_j^T;
//    once the tile's warpgroup has turned S into P = exp2(s * scale * log2 e - lse * log2 e)
//    in its registers, dP_t = dO_t V_j^T overwrites it; the warpgroup then writes
//    dS = P * (dP - D) as 16-bit pairs into the buffer's first 64 columns, the A operand of
//    dQ_t += dS_t K_j (K MN-major), accumulated in the tile's own D TMEM columns over the
//    key blocks in ascending order;
//  * warp 9 issues dP_0(j) dP_1(j) dQ_0(j) S_0(j+1) dQ_1(j) S_1(j+1), so each tile's softmax
//    work runs while the tensor cores work on the other tile;
//  * warpgroup t (thread = query row = TMEM lane) does tile t's P and dS and its epilogue
//    (dQ * scale rounded to 16 bits, stored row by row).
#include "fa_internal.h"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

template <int D>
struct DqCfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr int TILE_BYTES = 128 * D * 2;  // 128 rows of Q, dO, K or V
  static constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 B
  // K_j is held until both dQ products of key block j are done, V_j only until the dP
  // products: separate rings, so V_{j+1} loads while dQ(j) and S(j+1) run
  static constexpr int KST = (D == 128) ? 2 : 4, VST = (D == 128) ? 1 : 3;
  static constexpr int STAGES = KST + VST;
  static constexpr int THREADS = 384;
  // registers after setmaxnreg: control warpgroup 88, the two tile warpgroups 208 each
  static constexpr int REG_CTRL = 88, REG_TILE = 208;
  static constexpr int REG_SPLIT = 128 * REG_CTRL + 256 * REG_TILE;
  static_assert(REG_SPLIT <= 384 * 168, "register split above the launch allocation");
  // shared memory: Q_0, Q_1, dO_0, dO_1, then the K / V ring
  static constexpr int OFF_Q = 0, OFF_DO = 2 * TILE_BYTES, OFF_KV = 4 * TILE_BYTES;
  // barriers: q_full, per tile {s_full, sd_free, dp_full, ds_ready, dq_done}, final, then
  // full / empty of the K slots followed by the V slots
  static constexpr int B_Q = 0, B_TILE = 1 /*[5][2]*/, B_FINAL = 11, B_KV = 12 /*[2][STAGES]*/;
  static constexpr int NBARS = 12 + 2 * STAGES;
  static constexpr int SMEM = 1024 + OFF_KV + STAGES * TILE_BYTES + 8 * NBARS + 64;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM: tile t's S / dP / dS buffer at 128 t, its dQ accumulator at 256 + D t
  static constexpr uint32_t T_SD = 0, T_DQ = 256, TMEM_COLS = 512;
};

__device__ __forceinline__ float dq_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(384, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw_dq[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_dq) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_KV + C::STAGES * C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]

  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0 + 8u * C::B_Q, final_bar = bar0 + 8u * C::B_FINAL;
  auto tb = [&](int kind, int t) { return bar0 + 8u * (C::B_TILE + 2 * kind + t); };
  auto s_full = [&](int t) { return tb(0, t); };    // S_t ready (MMA commit)
  auto sd_free = [&](int t) { return tb(1, t); };   // S_t read into registers (128 threads)
  auto dp_full = [&](int t) { return tb(2, t); };   // dP_t ready (MMA commit)
  auto ds_ready = [&](int t) { return tb(3, t); };  // dS_t written (128 threads)
  auto dq_done = [&](int t) { return tb(4, t); };   // last dQ_t product done (MMA commit)
  // ring slot st: K slots 0 .. KST-1, V slots KST .. STAGES-1
  auto kv_full = [&](int st) { return bar0 + 8u * (C::B_KV + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (C::B_KV + C::STAGES + st); };
  // the c-th use of a ring (K: c = j, V: c = j): its slot and its phase on that slot
  auto kslot = [&](int j) { return j % C::KST; };
  auto vslot = [&](int j) { return C::KST + j % C::VST; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work decode: CTA = (batch, query head, 256 queries); with the mask, the units with
  // most key blocks first; query heads of a GQA group adjacent
  const int N = p.N;
  const int nqu = (N + 255) / 256;
  const int BH = p.B * p.Hq;
  int qu, bh;
  if (CAUSAL) {
    qu = nqu - 1 - static_cast<int>(blockIdx.x / BH);
    bh = static_cast<int>(blockIdx.x % BH);
  } else {
    qu = static_cast<int>(blockIdx.x % nqu);
    bh = static_cast<int>(blockIdx.x / nqu);
  }
  const int h = bh % p.Hq, b = bh / p.Hq;
  const int hkv = h / (p.Hq / p.Hkv);
  auto r0_of = [&](int t) { return 256 * qu + 128 * t; };
  // key blocks of tile t (keys past N are zero rows of K and V, so their dS K terms vanish)
  auto n_of = [&](int t) { return r0_of(t) >= N ? 0 : (CAUSAL ? r0_of(t) / 128 + 1 : (N + 127) / 128); };
  const int n0 = n_of(0), n1 = n_of(1);
  const int nmax = n0 > n1 ? n0 : n1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    wg_fail[0] = wg_fail[1] = 0;
    mbar_init(q_full, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(sd_free(t), 128);
      mbar_init(dp_full(t), 1);
      mbar_init(ds_ready(t), 128);
      mbar_init(dq_done(t), 1);
    }
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
    setmaxnreg_dec<C::REG_CTRL>();
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
        mbar_arrive_expect_tx(q_full, ((n0 > 0) + (n1 > 0)) * 2 * C::TILE_BYTES);
        for (int t = 0; t < 2; ++t) {
          if ((t ? n1 : n0) == 0) continue;
          for (int ch = 0; ch < C::CHUNKS; ++ch) {
            for (int half = 0; half < 2; ++half) {
              const int off = t * C::TILE_BYTES + ch * C::CHUNK_BYTES + half * 8192;
              tma_load_4d(smem_u32(smem + C::OFF_Q + off), &p.tm_q, q_full, ch * 64, h, r0_of(t) + 64 * half, b);
              tma_load_4d(smem_u32(smem + C::OFF_DO + off), &p.tm_do, q_full, ch * 64, h, r0_of(t) + 64 * half, b);
            }
          }
        }
      }
      bool ok = true;
      int nk = 0, nv = 0;  // K and V loads issued
      for (int j = 0; j < nmax && ok; ++j) {
        for (int kind = 0; kind < 2; ++kind) {  // K_j then V_j
          const int ns = kind ? C::VST : C::KST;
          const int slot = kind ? vslot(j) : kslot(j);
          if (j >= ns && !__all_sync(FULL, mbar_wait(kv_empty(slot), ((j / ns) - 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(kv_full(slot), C::TILE_BYTES);
            const CUtensorMap* map = kind ? &p.tm_v : &p.tm_k;
            for (int ch = 0; ch < C::CHUNKS; ++ch)
              tma_load_4d(smem_u32(smem + C::OFF_KV + slot * C::TILE_BYTES + ch * C::CHUNK_BYTES), map, kv_full(slot),
                          ch * 64, hkv, 128 * j, b);
          }
          ++(kind ? nv : nk);
        }
      }
      if (!ok) {
        if (leader) fail();
        // let the loads in flight land before the CTA exits
        for (int i = (nk > C::KST ? nk - C::KST : 0); i < nk; ++i)
          mbar_wait(kv_full(kslot(i)), (i / C::KST) & 1, nullptr, lim);
        for (int i = (nv > C::VST ? nv - C::VST : 0); i < nv; ++i)
          mbar_wait(kv_full(vslot(i)), (i / C::VST) & 1, nullptr, lim);
        mbar_wait(q_full, 0, nullptr, lim);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t bf = BF16 ? 1u : 0u;
      constexpr uint32_t id_sp = idesc_f16(128, 128, bf, 0, 0);  // S, dP: both operands K-major
      constexpr uint32_t id_dq = idesc_f16(128, D, bf, 0, 1);    // dQ: K MN-major
      bool ok = __all_sync(FULL, mbar_wait(q_full, 0, abort_flag, lim));
      const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t ddo0 = smem_desc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
      const uint64_t dkv0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
      const uint64_t dk_mn0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), C::CHUNK_BYTES, 1024);
      auto u16 = [](int bytes) { return static_cast<uint64_t>(bytes >> 4); };
      // S_t(j) = Q_t K_j^T into tile t's buffer; issued right after dQ_t(j-1), the last
      // reader of that buffer, so each tile's chain S -> P -> dP -> dS -> dQ runs while the
      // tensor cores work on the other tile
      auto issue_s = [&](int t, int ks) {
        if (leader) {
#pragma unroll 1
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t o = u16((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32);
            mma_ss(tbase + C::T_SD + 128u * t, dq0 + u16(t * C::TILE_BYTES) + o, dkv0 + u16(ks * C::TILE_BYTES) + o,
                   id_sp, kk > 0 ? 1u : 0u);
          }
          mma_commit(s_full(t));
        }
      };
      auto wait_k = [&](int j) {
        if (!__all_sync(FULL, mbar_wait(kv_full(kslot(j)), (j / C::KST) & 1, abort_flag, lim))) return false;
        tc_fence_after();
        return true;
      };
      if (ok && nmax > 0) {
        ok = wait_k(0);
        if (ok) {
          if (n0 > 0) issue_s(0, kslot(0));
          if (n1 > 0) issue_s(1, kslot(0));
        }
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int ks = kslot(j), vs = vslot(j);
        // dP_t = dO_t V_j^T over S_t, once tile t's warpgroup holds S_t in registers
        if (!__all_sync(FULL, mbar_wait(kv_full(vs), (j / C::VST) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= (t ? n1 : n0)) continue;
          if (!__all_sync(FULL, mbar_wait(sd_free(t), j & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
#pragma unroll 1
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t o = u16((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32);
              mma_ss(tbase + C::T_SD + 128u * t, ddo0 + u16(t * C::TILE_BYTES) + o,
                     dkv0 + u16(vs * C::TILE_BYTES) + o, id_sp, kk > 0 ? 1u : 0u);
            }
            mma_commit(dp_full(t));
          }
        }
        if (!ok) break;
        if (leader) mma_commit(kv_empty(vs));  // V_j is read only by the dP products
        // dQ_t += dS_t K_j: dS from TMEM (16-bit pairs, keys 2i, 2i+1 in column i), K MN-major;
        // then S_t(j+1)
        bool k_next = false;
        const int t_last = j < n1 ? 1 : 0;  // the last tile that reads K_j
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nt = t ? n1 : n0;
          if (j >= nt) continue;
          if (!__all_sync(FULL, mbar_wait(ds_ready(t), j & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint64_t kd = dk_mn0 + u16(ks * C::TILE_BYTES);
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tbase + C::T_DQ + uint32_t(D) * t, tbase + C::T_SD + 128u * t + 8u * kk, kd + u16(kk * 2048),
                     id_dq, (j > 0 || kk > 0) ? 1u : 0u);
            if (j == nt - 1) mma_commit(dq_done(t));
            if (t == t_last) mma_commit(kv_empty(ks));  // K_j: read by S and dQ
          }
          if (j + 1 < nt) {
            if (!k_next && !(k_next = wait_k(j + 1))) {
              ok = false;
              break;
            }
            issue_s(t, kslot(j + 1));
          }
        }
        if (!ok) break;
      }
      if (!ok && leader) fail();
      if (leader) mma_commit(final_bar);
      mbar_wait(final_bar, 0, nullptr, lim);
      // the last commits to kv_empty have no consumer: let them land before exit
      if (ok) {
        for (int i = (nmax > C::KST ? nmax - C::KST : 0); i < nmax; ++i)
          mbar_wait(kv_empty(kslot(i)), (i / C::KST) & 1, nullptr, lim);
        for (int i = (nmax > C::VST ? nmax - C::VST : 0); i < nmax; ++i)
          mbar_wait(kv_empty(vslot(i)), (i / C::VST) & 1, nullptr, lim);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<C::REG_TILE>();
    // ------------------------------------------------------- tile warpgroups
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int row = r0_of(t) + r;
    const int nt = t ? n1 : n0;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t sd_tm = tbase + lane_off + C::T_SD + 128u * t;
    const float cl2 = p.scale_log2;
    // -lse * log2(e) and -D of this query row, from the preprocess (-inf and 0 past N)
    const long long vrow = static_cast<long long>(bh) * p.Npad + row;
    const float nl2 = row < p.Npad ? p.l2vec[vrow] : -INFINITY;
    const float nd = row < p.Npad ? p.dvec[vrow] : 0.f;
    const uint64_t cl2x2 = f2pack(cl2, cl2), nl2x2 = f2pack(nl2, nl2), ndx2 = f2pack(nd, nd);
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!__all_sync(FULL, mbar_wait(s_full(t), j & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float pv[128];
      {
        uint32_t* sv = reinterpret_cast<uint32_t*>(pv);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(sd_tm + 32u * c, sv + 32 * c);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(sd_free(t));  // dP_t may now overwrite S_t
      // P = exp2(s * scale * log2 e - lse * log2 e), masked on the diagonal block
      const int nvis = (CAUSAL && j == nt - 1) ? row + 1 - 128 * j : 128;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        float a0, a1;
        f2unpack(ffma2(f2pack(pv[c], pv[c + 1]), cl2x2, nl2x2), a0, a1);
        pv[c] = dq_ex2(a0);
        pv[c + 1] = dq_ex2(a1);
        if (CAUSAL) {
          if (c >= nvis) pv[c] = 0.f;
          if (c + 1 >= nvis) pv[c + 1] = 0.f;
        }
      }
      if (!__all_sync(FULL, mbar_wait(dp_full(t), j & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dS = P (dP - D), 32 keys at a time: keys [32 c, 32 c + 32) go as 16 packed columns to
      // [16 c, 16 c + 16), which this thread has already read
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t dpv[32];
        tmem_ld32(sd_tm + 32u * c, dpv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          float d0, d1;
          f2unpack(fmul2(f2pack(pv[32 * c + 2 * u], pv[32 * c + 2 * u + 1]),
                         fadd2(f2pack(__uint_as_float(dpv[2 * u]), __uint_as_float(dpv[2 * u + 1])), ndx2)),
                   d0, d1);
          pk[u] = pack_half2<BF16>(d0, d1);
        }
        tmem_st16(sd_tm + 16u * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_ready(t));
    }
    if (nt > 0) {
      if (ok && !mbar_wait(dq_done(t), 0, abort_flag, lim)) ok = false;
      if (!ok) {
        wg_fail[t] = 1;
        fail();
      }
      named_bar_sync_n(1 + t, 128);
      if (wg_fail[t] == 0) {  // uniform across the warpgroup
        tc_fence_after();
        uint16_t* out = p.dq + ((static_cast<long long>(b) * N + row) * p.Hq + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + C::T_DQ + uint32_t(D) * t + 32u * c, v);  // all lanes (.sync.aligned)
          tmem_wait_ld();
          if (row >= N) continue;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 o;
            o.x = pack_half2<BF16>(__uint_as_float(v[8 * u + 0]) * p.scale, __uint_as_float(v[8 * u + 1]) * p.scale);
            o.y = pack_half2<BF16>(__uint_as_float(v[8 * u + 2]) * p.scale, __uint_as_float(v[8 * u + 3]) * p.scale);
            o.z = pack_half2<BF16>(__uint_as_float(v[8 * u + 4]) * p.scale, __uint_as_float(v[8 * u + 5]) * p.scale);
            o.w = pack_half2<BF16>(__uint_as_float(v[8 * u + 6]) * p.scale, __uint_as_float(v[8 * u + 7]) * p.scale);
            *reinterpret_cast<uint4*>(out + 32 * c + 8 * u) = o;
          }
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
  cudaError_t e = prepare_launch_once<fa_bwd_dq_kernel<D, BF16, CAUSAL>>(C::SMEM, C::THREADS, C::REG_SPLIT);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((p.N + 255) / 256) * p.B * p.Hq;
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
