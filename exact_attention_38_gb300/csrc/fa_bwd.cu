// Backward pass of exact attention on sm_103a: dQ, dK, dV of L = sum(dO * O).
//
// The pages ask for gradients equal to the plain definition's within tolerance
// ("FlashAttention-2: atención eficiente en GPU para contextos largos", section
// "Bloques pequeños, normalización global") and a backward "almost as fast as the
// forward" with MQA/GQA ("FlashAttention-T: Optimización GPU para LLMs Escalables",
// section "Innovaciones técnicas frente a FlashAttention original").  The pass is the
// textbook gradient evaluated tile by tile, recomputing P from the saved log-sum-exp
// instead of storing it:
//
//   D_i    = <dO_i, O_i>                                   (fa_bwd_preprocess)
//   P_ij   = exp(scale * q_i.k_j - lse_i)
//   dV_j  += sum_i P_ij dO_i
//   dS_ij  = P_ij (dO_i.v_j - D_i)
//   dK_j  += scale * sum_i dS_ij q_i
//   dQ_i  += scale * sum_j dS_ij k_j                       (fp32 workspace, then fa_bwd_dq_convert)
//
// fa_bwd_main: one CTA per (batch, key/value head, block of 128 keys).  K_j and V_j stay
// in shared memory; the CTA walks every query head of its GQA group and every visible
// block of 64 queries.  Per step the tensor cores compute S^T = K Q^T and dP^T = V dO^T
// into tensor memory (S^T double-buffered, V itself held in TMEM as the A operand);
// two softmax warpgroups (thread = key row = TMEM lane, each taking 32 of the 64 query
// columns) turn them into P^T and dS^T, both written back as 16-bit pairs into the S^T
// columns they read (dS^T also to swizzled shared memory); the tensor cores then accumulate
// dV += P^T dO and dK += dS^T Q in TMEM for the whole walk (A operands from TMEM) and
// compute dQ^T = K^T dS^T into the same S^T buffer, which a fourth warpgroup reads out
// and adds into the fp32 dQ accumulator while the next step's dP^T / S^T run: at d=128
// straight from registers (one coalesced reduction per query and warp: 32 consecutive d,
// 128 bytes); at d=64, where only two of its warps hold dQ^T rows, through a swizzled
// shared-memory tile and TMA tensor reductions (measured faster there).
// Taking operands from TMEM, and keeping the dQ^T additions out of shared memory, matters
// because the tensor cores read shared-memory operands at 128 B/clk per SM and every other
// shared-memory access competes with them.
// Without the mask, a last wave of key-block CTAs that would fill at most half the SMs is
// split: each of its key blocks runs as two CTAs over halves of the walk, which add fp32
// dK / dV partials that fa_bwd_split_convert then writes.  Short sequences run the same
// steps in the persistent kernel of fa_bwd_persist.cu.
#include "fa_internal.h"
#include "fa_bwd_common.cuh"
#include "sm100_ptx.cuh"

#include <cuda_fp16.h>

namespace fa {

template <int D>
struct BwdCfg {
  static constexpr int BK = 128;                  // keys per CTA (TMEM lanes)
  static constexpr int BQ = 64;                   // queries per step
  static constexpr int CHUNKS = D / 64;           // 128-byte swizzle column chunks
  static constexpr int KV_TILE = 128 * D * 2;     // K or V tile
  static constexpr int KV_CHUNK = 128 * 128;      // 128 rows x 128 B
  static constexpr int Q_CHUNK = 64 * 128;        // 64 rows x 128 B
  static constexpr int Q_TILE = 64 * D * 2;       // Q or dO tile
  static constexpr int DS_TILE = 128 * 64 * 2;    // dS^T tile, 128 keys x 64 queries, 16-bit
  static constexpr int STG = (D == 128) ? 4 : 6;  // Q/dO/lse/D stages
  static constexpr int THREADS = 512;
  // barrier indices
  // dq_full has one barrier per dQ^T buffer: with a single one the MMA could complete the
  // phases of two consecutive steps before the dQ warpgroup polls the first of them, and
  // the parity it then sees would look unchanged
  static constexpr int B_KV = 0, B_SDP = 1, B_DPFREE = 2, B_DSREADY = 3 /*[2]*/, B_DSFREE = 5 /*[2]*/,
                       B_DQFULL = 7 /*[2]*/, B_DQFREE = 9, B_ACC = 10, B_FINAL = 11, B_VTM = 12,
                       B_STFULL = 13 /*[STG]*/;
  static constexpr int NBARS = 13 + 2 * STG;
  // shared-memory layout (offsets from the 1024-aligned base).  V is loaded into the
  // dS^T buffers, copied into TMEM, and never read from shared memory again.
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = KV_TILE;                        // [STG] Q tiles
  static constexpr int OFF_DO = OFF_Q + STG * Q_TILE;          // [STG] dO tiles
  static constexpr int OFF_DS = OFF_DO + STG * Q_TILE;         // [2] dS^T tiles (V first)
  static constexpr int OFF_V = OFF_DS;
  static_assert(2 * DS_TILE >= KV_TILE, "V fits in the dS^T buffers");
  // d=64: dQ^T staged as two [d rows x 32 fp32 queries] halves (128-byte rows, 128-byte
  // swizzle) for the TMA tensor reductions; d=128 adds from registers and stages nothing.
  // The fp32 accumulator is [B*Hq, Npad, d] at d=128 and [B*Hq, d, Npad] at d=64.
  static constexpr bool DQ_TMA = (D == 64);
  // MMA issue order of a step's two products (see the MMA warp)
  static constexpr bool DP_FIRST = (D == 128);
  static constexpr int DQ_HALF = D * 128;
  static constexpr int OFF_DQS = OFF_DS + 2 * DS_TILE;
  static constexpr int DQS_BYTES = DQ_TMA ? 2 * DQ_HALF : 0;
  static constexpr int OFF_LD = OFF_DQS + DQS_BYTES;           // [STG][2][64] floats: -lse*log2e, -D
  static constexpr int OFF_BAR = OFF_LD + STG * 2 * 64 * 4;
  // no alignment slack: the dynamic shared-memory base is 1024-byte aligned (checked at
  // run time by the kernel)
  static constexpr int SMEM = OFF_BAR + 8 * NBARS + 64;
  static_assert(SMEM <= 232448, "shared memory budget");
  // tensor-memory columns: S^T[2] (each later holding P^T | dS^T, then dQ^T), dP^T,
  // V (16-bit pairs, the A operand of dP^T), dV, dK
  static constexpr uint32_t T_S = 0, T_DP = 128, T_V = 192, T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
};

// ------------------------------------------------------------------- preprocess
// -D = -rowsum(dO * O) and -lse * log2(e) in the padded [B*Hq, Npad] layout (negated so
// the main kernel adds them; 0 and -inf past N, which zeroes P for padded query rows);
// zeroes the fp32 dQ accumulator.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess(const __grid_constant__ BwdParams p) {
  constexpr int LPR = D / 8;  // lanes per row, 8 elements (16 B) per lane
  const long long rows = static_cast<long long>(p.B) * p.N * p.Hq;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  // each warp keeps kGroups row groups of loads in flight before it reduces any
  constexpr int RPW = 32 / LPR, kGroups = 4;
  for (long long base = wid * RPW * kGroups; base < rows; base += warps_total * RPW * kGroups) {
    uint4 a[kGroups], g[kGroups];
#pragma unroll
    for (int u = 0; u < kGroups; ++u) {
      const long long r = base + u * RPW + sub;
      a[u] = g[u] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        a[u] = *reinterpret_cast<const uint4*>(p.o + r * D + part * 8);
        g[u] = *reinterpret_cast<const uint4*>(p.dout + r * D + part * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroups; ++u) {
      const long long r = base + u * RPW + sub;
      const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, gv[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        acc += bw_unpack_lo<BF16>(av[i]) * bw_unpack_lo<BF16>(gv[i]) +
               bw_unpack_hi<BF16>(av[i]) * bw_unpack_hi<BF16>(gv[i]);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (r < rows && part == 0) {
        // r = (b*N + n)*Hq + h
        const int h = static_cast<int>(r % p.Hq);
        const long long bn = r / p.Hq;
        const int n = static_cast<int>(bn % p.N);
        const int b = static_cast<int>(bn / p.N);
        const long long bh = static_cast<long long>(b) * p.Hq + h;
        p.dvec[bh * p.Npad + n] = -acc;
        p.l2vec[bh * p.Npad + n] = -p.lse[bh * p.N + n] * kLog2e;
      }
    }
  }
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  // padding entries n in [N, Npad)
  const int pad = p.Npad - p.N;
  const long long npad = static_cast<long long>(p.B) * p.Hq * pad;
  for (long long i = tid; i < npad; i += nthreads) {
    const long long bh = i / pad;
    const int n = p.N + static_cast<int>(i % pad);
    p.dvec[bh * p.Npad + n] = 0.f;
    p.l2vec[bh * p.Npad + n] = -INFINITY;
  }
  // dQ accumulator = 0 (16 B per thread per step); none when dQ is computed elsewhere
  const long long nacc4 = p.dq_acc ? static_cast<long long>(p.B) * p.Hq * D * p.Npad / 4 : 0;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long i = tid; i < nacc4; i += nthreads) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // wave-tail split: the fp32 dK / dV partials = 0
  const long long npart4 = static_cast<long long>(p.nsplit) * 2 * 128 * D / 4;
  float4* part4 = reinterpret_cast<float4*>(p.kv_part);
  for (long long i = tid; i < npart4; i += nthreads) part4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Variable-length form: rows (b*Hq + h, n) of the padded layout, n < Npad; query n of
// sequence b is packed row start_q + n.  A row whose lse is -inf (it sees no key) gets
// -inf as well, so its P is 0.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_varlen(const __grid_constant__ BwdParams p) {
  constexpr int LPR = D / 8;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Npad;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  for (long long base = wid * (32 / LPR); base < rows; base += warps_total * (32 / LPR)) {
    const long long r = base + sub;
    const long long bh = r / p.Npad;
    const int n = static_cast<int>(r % p.Npad);
    const int b = static_cast<int>(bh / p.Hq), h = static_cast<int>(bh % p.Hq);
    int sq = 0, lq = 0, sk = 0, lk = 0;
    const bool live = r < rows && seq_span(p.vl, b, sq, lq, sk, lk) && n < lq;
    float acc = 0.f;
    if (live) {
      const long long off = (static_cast<long long>(sq + n) * p.Hq + h) * D + part * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(p.o + off);
      const uint4 g = *reinterpret_cast<const uint4*>(p.dout + off);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        acc += bw_unpack_lo<BF16>(av[i]) * bw_unpack_lo<BF16>(gv[i]) +
               bw_unpack_hi<BF16>(av[i]) * bw_unpack_hi<BF16>(gv[i]);
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (r < rows && part == 0) {
      float l2 = -INFINITY;
      if (live) {
        const float lse = p.lse[static_cast<long long>(h) * p.vl.total_q + sq + n];
        l2 = lse == -INFINITY ? -INFINITY : -lse * kLog2e;
      }
      p.dvec[bh * p.Npad + n] = live ? -acc : 0.f;
      p.l2vec[bh * p.Npad + n] = l2;
    }
  }
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long nacc4 = static_cast<long long>(p.B) * p.Hq * D * p.Npad / 4;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long i = tid; i < nacc4; i += nthreads) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ dQ convert
// d=128: dQ[b, n, h, :] = scale * acc[b*Hq + h, n, :]: each thread converts 8 consecutive
// elements of one row (two 16-byte reads, one 16-byte write); consecutive threads walk
// the output in order, so the writes are contiguous and every read covers whole rows.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert(const __grid_constant__ BwdParams p) {
  constexpr int TPR = D / 8;  // threads per row
  const int nrow = VARLEN ? p.Npad : p.N;
  const long long total = static_cast<long long>(p.B) * nrow * p.Hq * TPR;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const long long row = i / TPR;  // (b * nrow + n) * Hq + h
    const int part = static_cast<int>(i % TPR);
    const int h = static_cast<int>(row % p.Hq);
    const long long bn = row / p.Hq;
    const int n = static_cast<int>(bn % nrow);
    const int b = static_cast<int>(bn / nrow);
    long long orow = static_cast<long long>(b) * p.N + n;  // output row of query n
    if (VARLEN) {
      int sq = 0, lq = 0, sk = 0, lk = 0;
      if (!seq_span(p.vl, b, sq, lq, sk, lk) || n >= lq) continue;
      orow = sq + n;
    }
    const float4* src =
        reinterpret_cast<const float4*>(p.dq_acc + (static_cast<long long>(b * p.Hq + h) * p.Npad + n) * D + 8 * part);
    const float4 a = src[0], c = src[1];
    const float sc = p.scale;
    uint4 o;
    o.x = pack_half2<BF16>(a.x * sc, a.y * sc);
    o.y = pack_half2<BF16>(a.z * sc, a.w * sc);
    o.z = pack_half2<BF16>(c.x * sc, c.y * sc);
    o.w = pack_half2<BF16>(c.z * sc, c.w * sc);
    *reinterpret_cast<uint4*>(p.dq + (orow * p.Hq + h) * D + 8 * part) = o;
  }
}

// d=64: dQ[b, n, h, :] = scale * acc[b*Hq + h, :, n]: a tiled transpose through shared
// memory (coalesced fp32 reads along n, coalesced 16-bit writes along d); one block per
// (b*Hq + h, 64 queries).
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_t(const __grid_constant__ BwdParams p) {
  __shared__ float tile[D][65];
  const int nblk = VARLEN ? p.Npad / 64 : (p.N + 63) / 64;
  const int bh = static_cast<int>(blockIdx.x / nblk);
  const int n0 = 64 * static_cast<int>(blockIdx.x % nblk);
  const int b = bh / p.Hq, h = bh % p.Hq;
  int len_q = p.N;
  long long row0 = static_cast<long long>(b) * p.N;  // output row of query 0 of this sequence
  if (VARLEN) {
    int sq = 0, sk = 0, lk = 0;
    if (!seq_span(p.vl, b, sq, len_q, sk, lk)) return;
    if (n0 >= len_q) return;
    row0 = sq;
  }
  const float* src = p.dq_acc + static_cast<long long>(bh) * D * p.Npad + n0;
#pragma unroll 8
  for (int i = threadIdx.x; i < D * 64; i += 256) {
    const int dd = i >> 6, n = i & 63;
    tile[dd][n] = src[static_cast<long long>(dd) * p.Npad + n];
  }
  __syncthreads();
  constexpr int G = D / 8;  // 8 outputs (16 B) per thread and step
  for (int i = threadIdx.x; i < 64 * G; i += 256) {
    const int n = i / G, g = i % G;
    if (n0 + n >= len_q) continue;
    uint4 o;
    o.x = pack_half2<BF16>(tile[8 * g + 0][n] * p.scale, tile[8 * g + 1][n] * p.scale);
    o.y = pack_half2<BF16>(tile[8 * g + 2][n] * p.scale, tile[8 * g + 3][n] * p.scale);
    o.z = pack_half2<BF16>(tile[8 * g + 4][n] * p.scale, tile[8 * g + 5][n] * p.scale);
    o.w = pack_half2<BF16>(tile[8 * g + 6][n] * p.scale, tile[8 * g + 7][n] * p.scale);
    *reinterpret_cast<uint4*>(p.dq + ((row0 + n0 + n) * p.Hq + h) * D + 8 * g) = o;
  }
}

// ------------------------------------------------------------- dK / dV epilogue
// Writes the 128-key tile held in TMEM columns [col, col + D) (thread r = key row r, fp32),
// times `mul`, as 16-bit rows.  Fixed length: through a shared-memory tile laid out as the
// K/V loads (64-column chunks of 128 rows x 128 B, 128-byte swizzle) and TMA tensor stores,
// which clip rows past N; the 128 threads of the calling warpgroup take part (named barrier
// `bar_id`).  Variable length: row by row (a tile store could run into the next sequence).
template <int D, bool BF16, bool VARLEN>
__device__ __forceinline__ void bwd_write_tile(uint32_t tm, float mul, uint8_t* stage, const CUtensorMap* map,
                                               uint16_t* out_row, bool live, int bar_id, int r, int hkv, int k0,
                                               int b) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tm + 32u * c, v);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_half2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
    if (VARLEN) {
      if (live) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(out_row + 32 * c + 8 * u) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    } else {
      uint8_t* rowp = stage + (c >> 1) * (128 * 128) + r * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = (c & 1) * 4 + u;
        *reinterpret_cast<uint4*>(rowp + ((unit ^ (r & 7)) * 16)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    }
  }
  if (!VARLEN) {
    fence_proxy_async_smem();
    named_bar_sync_n(bar_id, 128);
    if (r == 0) {
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) tma_store_4d(map, smem_u32(stage + ch * (128 * 128)), ch * 64, hkv, k0, b);
      bulk_commit_group();
      bulk_wait_group_read0();  // the staging must outlive the copy's reads of it
    }
  }
}

// Adds the fp32 128-key tile held in TMEM columns [col, col + D) (thread r = key row r) into
// tile `idx` of the wave-tail split's partials (tensor map over [2 nsplit][128][D] fp32):
// staged as 32-column chunks of 128 rows x 128 B (128-byte swizzle), then one TMA tensor
// reduction per chunk; the 128 threads of the calling warpgroup take part (named barrier
// `bar_id`).
template <int D>
__device__ __forceinline__ void bwd_add_partial(uint32_t tm, uint8_t* stage, const CUtensorMap* map, int idx,
                                                int bar_id, int r) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tm + 32u * c, v);
    tmem_wait_ld();
    uint8_t* rowp = stage + c * (128 * 128) + r * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
  fence_proxy_async_smem();
  named_bar_sync_n(bar_id, 128);
  if (r == 0) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) tma_reduce_add_3d(map, smem_u32(stage + c * (128 * 128)), 32 * c, 0, idx);
    bulk_commit_group();
    bulk_wait_group_read0();  // the staging must outlive the reductions' reads of it
  }
}

// dk / dv of the wave-tail split's key blocks: the sum of the two halves' fp32 partials,
// dK times the scale, rounded to 16 bits.  One thread per 8 columns of a row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_split_convert(const __grid_constant__ BwdParams p) {
  constexpr int G8 = D / 8;
  const int nkb = (p.N + 127) / 128;
  const long long total = static_cast<long long>(p.nsplit) * 2 * 128 * G8;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int g8 = static_cast<int>(i % G8);
    const int row = static_cast<int>((i / G8) % 128);
    const int tile = static_cast<int>(i / (G8 * 128));  // 2 * split + (0: dK, 1: dV)
    const int unit = p.split_first + tile / 2;
    const int jb = unit % nkb, bhk = unit / nkb;
    const int key = 128 * jb + row;
    if (key >= p.N) continue;
    const float* src = p.kv_part + (static_cast<long long>(tile) * 128 + row) * D + 8 * g8;
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 c = *reinterpret_cast<const float4*>(src + 4);
    const float mul = (tile & 1) ? 1.0f : p.scale;
    uint4 o;
    o.x = pack_half2<BF16>(a.x * mul, a.y * mul);
    o.y = pack_half2<BF16>(a.z * mul, a.w * mul);
    o.z = pack_half2<BF16>(c.x * mul, c.y * mul);
    o.w = pack_half2<BF16>(c.z * mul, c.w * mul);
    uint16_t* out = (tile & 1) ? p.dv : p.dk;
    const int hkv = bhk % p.Hkv, b = bhk / p.Hkv;
    *reinterpret_cast<uint4*>(out + ((static_cast<long long>(b) * p.N + key) * p.Hkv + hkv) * D + 8 * g8) = o;
  }
}

// ------------------------------------------------------------------- main kernel
template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool DQ>
__global__ void __launch_bounds__(512, 1) fa_bwd_main(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_bwd[];
  // the 128-byte-swizzled tiles need 1024-byte alignment; with a misaligned base the
  // kernel records an error and does nothing (uniform early exit, before any barrier)
  if ((smem_u32(smem_bwd) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kDevErrLayout);
    return;
  }
  uint8_t* smem = smem_bwd;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wg_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [4]
  volatile int* dq_fail = reinterpret_cast<volatile int*>(tmem_slot + 6);  // d=64 dQ warps gave up
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * i; };
  const uint32_t kv_full = bar(C::B_KV), sdp_full = bar(C::B_SDP), dp_free = bar(C::B_DPFREE);
  const uint32_t dq_free = bar(C::B_DQFREE), acc_done = bar(C::B_ACC);
  const uint32_t final_bar = bar(C::B_FINAL), v_tmem = bar(C::B_VTM);
  auto ds_ready = [&](int b) { return bar(C::B_DSREADY + b); };
  auto ds_free = [&](int b) { return bar(C::B_DSFREE + b); };
  auto dq_full = [&](int b) { return bar(C::B_DQFULL + b); };
  auto st_full = [&](int s) { return bar(C::B_STFULL + s); };
  auto st_empty = [&](int s) { return bar(C::B_STFULL + C::STG + s); };
  constexpr unsigned FULL = 0xffffffffu;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work decode: key blocks of one (batch, key/value head) are consecutive CTAs
  // (ascending, so with the causal mask the heaviest come first); the CTAs resident
  // at any time then share a few heads' Q, dO and dQ accumulator through L2.  With the
  // mask, a fixed length of at least 32 key blocks and at most 64 (batch, key/value head)
  // pairs, key block jb of every head comes before jb + 1 of any: heaviest first over the
  // whole grid, which balances the last wave better (measured: 16k tokens 2.25 -> 2.19 ms,
  // GQA 32 / 8 heads 4.55 -> 4.40); with more, shorter heads the head-by-head order wins.
  const int N = VARLEN ? p.vl.max_k : p.N;  // key rows the grid covers per sequence
  const int nkb = (N + 127) / 128;
  const int BHK = p.B * p.Hkv;
  const bool kb_major = CAUSAL && !VARLEN && nkb >= 32 && BHK <= 64;
  // Wave-tail split (fixed length, non-causal): the grid's last nsplit key blocks would
  // run on a fraction of the SMs after the others are done, so each runs as two CTAs,
  // half of the query walk each (half = 0, 1; -1 for a whole walk).
  int unit = static_cast<int>(blockIdx.x), half = -1;
  if (!CAUSAL && !VARLEN && p.nsplit > 0 && unit >= p.split_first) {
    half = (unit - p.split_first) & 1;
    unit = p.split_first + ((unit - p.split_first) >> 1);
  }
  const int jb = kb_major ? unit / BHK : unit % nkb;
  const int bhk = kb_major ? unit % BHK : unit / nkb;
  const int hkv = bhk % p.Hkv;
  const int b = bhk / p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int k0 = 128 * jb;
  // Sequence geometry (fixed length: len_q = len_k = N).  With variable lengths and the
  // mask, query i sees key j iff j <= i + (len_k - len_q), so the first query block
  // that sees key k0 is (k0 - off) / 64.
  int start_q = 0, len_q = N, start_k = 0, len_k = N;
  if (VARLEN) {
    if (!seq_span(p.vl, b, start_q, len_q, start_k, len_k)) {
      if (threadIdx.x == 0 && jb == 0 && hkv == 0) atomicOr(p.err, kDevErrSeqlens);
      return;  // uniform, before any barrier or TMEM allocation
    }
    if (k0 >= len_k) return;
  }
  const int off = len_k - len_q;
  const int nqb = (len_q + 63) / 64;
  const int qb0 = CAUSAL ? (VARLEN ? max(0, k0 - off) / 64 : 2 * jb) : 0;
  const int nq = max(0, nqb - qb0);  // query blocks per head
  // steps [it0, it0 + T) of the walk over G * nq (query head, query block) steps
  const int it0 = half == 1 ? G * nq / 2 : 0;
  const int T = half < 0 ? G * nq : (half == 0 ? G * nq / 2 : G * nq - G * nq / 2);
  if (VARLEN && T == 0) {
    // no query sees these keys: dK = dV = 0
    for (int i = threadIdx.x; i < 128 * (D / 8); i += blockDim.x) {
      const int key = k0 + i / (D / 8);
      if (key >= len_k) continue;
      const long long o = (static_cast<long long>(start_k + key) * p.Hkv + hkv) * D + 8 * (i % (D / 8));
      *reinterpret_cast<uint4*>(p.dk + o) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(p.dv + o) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    wg_fail[0] = wg_fail[1] = wg_fail[2] = wg_fail[3] = 0;
    *dq_fail = 0;
    mbar_init(kv_full, 1);
    mbar_init(sdp_full, 1);
    mbar_init(dp_free, 256);
    mbar_init(ds_ready(0), 256);
    mbar_init(ds_ready(1), 256);
    mbar_init(ds_free(0), 1);
    mbar_init(ds_free(1), 1);
    mbar_init(dq_full(0), 1);
    mbar_init(dq_full(1), 1);
    mbar_init(dq_free, 128);
    mbar_init(acc_done, 1);
    mbar_init(final_bar, 1);
    mbar_init(v_tmem, 128);
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
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.err, kDevErrTimeout);
  };
  const int wg = warp >> 2;                        // 0,1: softmax; 2: dQ; 3: control
  const int r = (warp & 3) * 32 + lane;            // TMEM lane: key row (wg 0,1) or d index (wg 2)
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;

  if (wg == 3) {
    // launch allocation 512 x 128 registers: control 80, dQ 112, softmax 2 x 160
    setmaxnreg_dec<80>();
    // The control warps run their loops with all 32 lanes (warp-uniform control flow,
    // so loop state and descriptors live in uniform registers); one elected lane issues
    // the copies, the tcgen05 instructions and their commits.
    const bool leader = elect_one();
    if (warp == 12) {
      // ------------------------------------------------------------ TMA producer
      if (leader) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_do);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        if (C::DQ_TMA && DQ) tma_prefetch_desc(&p.tm_dq);
        if (!VARLEN) {
          tma_prefetch_desc(&p.tm_dk);
          tma_prefetch_desc(&p.tm_dv);
        }
        mbar_arrive_expect_tx(kv_full, 2 * C::KV_TILE);
        for (int ch = 0; ch < C::CHUNKS; ++ch) {
          if (VARLEN) {
            tma_load_3d(sbase + C::OFF_K + ch * C::KV_CHUNK, &p.tm_k, kv_full, ch * 64, hkv, start_k + k0);
            tma_load_3d(sbase + C::OFF_V + ch * C::KV_CHUNK, &p.tm_v, kv_full, ch * 64, hkv, start_k + k0);
          } else {
            tma_load_4d(sbase + C::OFF_K + ch * C::KV_CHUNK, &p.tm_k, kv_full, ch * 64, hkv, k0, b);
            tma_load_4d(sbase + C::OFF_V + ch * C::KV_CHUNK, &p.tm_v, kv_full, ch * 64, hkv, k0, b);
          }
        }
      }
      bool ok = true;
      int it = 0;
      for (; it < T; ++it) {
        const int s = it % C::STG;
        if (it >= C::STG &&
            !__all_sync(FULL, mbar_wait(st_empty(s), ((it / C::STG) - 1) & 1, abort_flag, lim))) {
          ok = false;
          break;
        }
        const int hq = hkv * G + (it0 + it) / nq;
        const int q0 = 64 * (qb0 + (it0 + it) % nq);
        if (leader) {
          mbar_arrive_expect_tx(st_full(s), 2 * C::Q_TILE + 2 * 256);
          for (int ch = 0; ch < C::CHUNKS; ++ch) {
            const uint32_t dq_ = sbase + C::OFF_Q + s * C::Q_TILE + ch * C::Q_CHUNK;
            const uint32_t ddo = sbase + C::OFF_DO + s * C::Q_TILE + ch * C::Q_CHUNK;
            if (VARLEN) {
              tma_load_3d(dq_, &p.tm_q, st_full(s), ch * 64, hq, start_q + q0);
              tma_load_3d(ddo, &p.tm_do, st_full(s), ch * 64, hq, start_q + q0);
            } else {
              tma_load_4d(dq_, &p.tm_q, st_full(s), ch * 64, hq, q0, b);
              tma_load_4d(ddo, &p.tm_do, st_full(s), ch * 64, hq, q0, b);
            }
          }
          const long long row = (static_cast<long long>(b) * p.Hq + hq) * p.Npad + q0;
          bulk_load(sbase + C::OFF_LD + s * 512, p.l2vec + row, 256, st_full(s));
          bulk_load(sbase + C::OFF_LD + s * 512 + 256, p.dvec + row, 256, st_full(s));
        }
      }
      if (!ok) {
        if (leader) fail();
        for (int i = (it > C::STG ? it - C::STG : 0); i < it; ++i)
          mbar_wait(st_full(i % C::STG), (i / C::STG) & 1, nullptr, lim);
        mbar_wait(kv_full, 0, nullptr, lim);
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
      bool ok = __all_sync(FULL, mbar_wait(kv_full, 0, abort_flag, lim) && mbar_wait(v_tmem, 0, abort_flag, lim));
      for (int it = 0; it <= T && ok; ++it) {
        if (it < T) {
          const int s = it % C::STG, bb = it & 1;
          if (!__all_sync(FULL, mbar_wait(st_full(s), (it / C::STG) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          const uint64_t qs = u16(s * C::Q_TILE);
          // S^T(it) overwrites the buffer that held dQ^T(it-2), which must have been read
          // out; dP^T(it) overwrites the columns the previous step's softmax has loaded.
          auto issue_s = [&]() {
            if (DQ && it >= 2 && !__all_sync(FULL, mbar_wait(dq_free, (it - 2) & 1, abort_flag, lim))) return false;
            tc_fence_after();
            // S^T = K Q^T  (both K-major in shared memory)
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tbase + C::T_S + 64u * bb, dK_km + u16((kk / 4) * C::KV_CHUNK + (kk % 4) * 32),
                       dQ_km + qs + u16((kk / 4) * C::Q_CHUNK + (kk % 4) * 32), id_sdp, kk > 0);
            }
            return true;
          };
          auto issue_dp = [&]() {
            if (it > 0 && !__all_sync(FULL, mbar_wait(dp_free, (it - 1) & 1, abort_flag, lim))) return false;
            tc_fence_after();
            // dP^T = V dO^T  (V from TMEM as 16-bit pairs; dO K-major)
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ts(tbase + C::T_DP, tbase + C::T_V + 8u * kk,
                       dDO_km + qs + u16((kk / 4) * C::Q_CHUNK + (kk % 4) * 32), id_sdp, kk > 0);
            }
            return true;
          };
          // Issue order, measured per head dimension on GB300: at d=128 dP^T first (it runs
          // while the dQ warpgroup reads dQ^T(it-2) out of S^T's buffer; 4.29 against 4.51 ms
          // for the 16k-token backward), at d=64 S^T first (6.48 against 6.78 ms).
          const bool issued = C::DP_FIRST ? (issue_dp() && issue_s()) : (issue_s() && issue_dp());
          if (!issued) {
            ok = false;
            break;
          }
          if (leader) mma_commit(sdp_full);  // covers both products
        }
        if (it > 0) {
          const int i = it - 1, s = i % C::STG, bb = i & 1;
          if (!__all_sync(FULL, mbar_wait(ds_ready(bb), (i >> 1) & 1, abort_flag, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qs = u16(s * C::Q_TILE), dss = u16(bb * C::DS_TILE);
          if (leader) {
            // k-step kk covers queries [16 kk, 16 kk + 16): in the S^T buffer, queries
            // [32 h, 32 h + 32) hold P^T in columns [32 h, 32 h + 16) and dS^T in
            // [32 h + 16, 32 h + 32), as 16-bit pairs
            // dV += P^T dO   (P^T from TMEM; dO MN-major: queries x d)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tbase + C::T_DV, tbase + C::T_S + 64u * bb + 32u * (kk / 2) + 8u * (kk % 2),
                     dDO_mn + qs + u16(kk * 2048), id_grad, (i > 0 || kk > 0));
            // dK += dS^T Q   (dS^T from TMEM; Q MN-major)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(tbase + C::T_DK, tbase + C::T_S + 64u * bb + 32u * (kk / 2) + 16u + 8u * (kk % 2),
                     dQ_mn + qs + u16(kk * 2048), id_grad, (i > 0 || kk > 0));
            // the stage's Q / dO are no longer read once these complete
            mma_commit(st_empty(s));
          }
          if (leader) {
            // dQ^T = K^T dS^T into the step's S^T buffer, after dV and dK above have read
            // P^T and dS^T from it (tcgen05.mma executes in issue order).  K^T: MN-major
            // view of the K tile, d padded to 128 rows; dS^T: MN-major, queries contiguous.
            if (DQ) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tbase + C::T_S + 64u * bb, dK_mn + u16(kk * 2048), dDS_mn + dss + u16(kk * 2048), id_dq,
                       kk > 0);
              mma_commit(dq_full(bb));
            }
            mma_commit(ds_free(bb));
          }
        }
      }
      if (!ok && leader) fail();
      if (leader) {
        mma_commit(acc_done);
        mma_commit(final_bar);
      }
      mbar_wait(final_bar, 0, nullptr, lim);
      // The last commits to st_empty and ds_free have no consumer; let their arrivals land
      // before this CTA's shared memory (and the barriers in it) passes to the next CTA.
      if (ok) {
        for (int i = (T > C::STG ? T - C::STG : 0); i < T; ++i)
          mbar_wait(st_empty(i % C::STG), (i / C::STG) & 1, nullptr, lim);
        for (int i = (T > 2 ? T - 2 : 0); i < T; ++i) mbar_wait(ds_free(i & 1), (i >> 1) & 1, nullptr, lim);
      }
      __syncwarp();
    }
  } else if (wg < 2) {
    setmaxnreg_inc<160>();
    // ------------------------------------------------------ P^T and dS^T
    // warpgroup wg takes query columns [32 wg, 32 wg + 32) of each 64-column step
    bool ok = true;
    const float cl2 = p.scale_log2;
    const uint64_t cl2x2 = f2pack(cl2, cl2);
    const int key = k0 + r;
    const int cbase = 32 * wg;
    if (wg == 0) {
      // V row r -> TMEM lane r as 16-bit pairs (the A operand of dP^T = V dO^T); V's
      // shared-memory copy sits in the dS^T buffers, which are written only after this
      if (!__all_sync(FULL, mbar_wait(kv_full, 0, abort_flag, lim))) {
        ok = false;
      } else {
        bwd_v_to_tmem<C::CHUNKS>(smem + C::OFF_V, r, tbase + lane_off + C::T_V);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(v_tmem);
      }
    } else if (!__all_sync(FULL, mbar_wait(v_tmem, 0, abort_flag, lim))) {
      ok = false;  // warpgroup 1 writes dS^T over V's shared-memory copy: wait for the copy
    }
    for (int it = 0; it < T && ok; ++it) {
      const int s = it % C::STG, bb = it & 1;
      const int q0 = 64 * (qb0 + (it0 + it) % nq);
      if (!__all_sync(FULL, mbar_wait(st_full(s), (it / C::STG) & 1, abort_flag, lim) &&
                                mbar_wait(sdp_full, it & 1, abort_flag, lim))) {
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
      // per query column: -lse*log2(e) and -D, staged by the producer (float4 loads, the
      // same address in every lane)
      const float4* nl4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512) + cbase / 4;
      const float4* nd4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512 + 256) + cbase / 4;
      // with the causal mask query column c sees this key iff c >= key - off - q0; with
      // variable lengths a key past the sequence is seen by no column
      const int cmin = (VARLEN && key >= len_k) ? (1 << 20) : (CAUSAL ? key - off - q0 - cbase : -(1 << 20));
      // the dS^T buffer of this parity must have been consumed by the MMAs of step it-2
      if (it >= 2 && !__all_sync(FULL, mbar_wait(ds_free(bb), ((it >> 1) - 1) & 1, abort_flag, lim))) {
        ok = false;
        break;
      }
      // dS^T row r -> 128-byte swizzled row of the [128 keys x 64 queries] tile; this
      // warpgroup writes 16-byte units [4 wg, 4 wg + 4)
      uint8_t* rowp = smem + C::OFF_DS + bb * C::DS_TILE + r * 128;
      uint32_t pk[16], dsk[16];
      bwd_p_ds<BF16, CAUSAL || VARLEN, DQ>(sv, dpv, nl4, nd4, cmin, cl2x2, rowp, wg, r, pk, dsk);
      // P^T (16 packed columns) then dS^T (16) go back into the 32 columns of S^T this
      // warpgroup read, so neither warpgroup writes columns the other still reads
      tmem_st16(tbase + lane_off + C::T_S + 64u * bb + cbase, pk);
      tmem_st16(tbase + lane_off + C::T_S + 64u * bb + cbase + 16u, dsk);
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(ds_ready(bb));
    }
    // ---- epilogue (warpgroup 0): scale * dK -> 16-bit rows
    if (!ok) {
      wg_fail[wg] = 1;
      fail();
    }
    if (wg == 0) {
      if (!mbar_wait(acc_done, 0, abort_flag, lim)) {
        wg_fail[0] = 1;
        fail();
      }
      named_bar_sync_n(2, 128);
      if (wg_fail[0] == 0) {
        tc_fence_after();
        if (half >= 0) {
          bwd_add_partial<D>(tbase + lane_off + C::T_DK, smem + C::OFF_Q, &p.tm_kvpart, 2 * (unit - p.split_first), 2,
                             r);
        } else {
          const long long krow = VARLEN ? static_cast<long long>(start_k) + key : static_cast<long long>(b) * N + key;
          bwd_write_tile<D, BF16, VARLEN>(tbase + lane_off + C::T_DK, p.scale, smem + C::OFF_Q, &p.tm_dk,
                                          p.dk + (krow * p.Hkv + hkv) * D, key < len_k, 2, r, hkv, k0, b);
        }
      }
    }
  } else {
    setmaxnreg_dec<112>();
    // ------------------------------------------- dQ^T -> fp32 accumulator
    // Thread r holds row d = r of dQ^T (64 query columns).  Once they are in registers the
    // TMEM buffer is released, and they are added into the fp32 accumulator.  d=128
    // ([B*Hq, Npad, d], d contiguous): one reduction per query, the 32 lanes of a warp
    // covering 32 consecutive d (one aligned 128-byte line).  d=64 ([B*Hq, d, Npad], queries
    // contiguous): each 32-query half is staged as [d rows x 128 B] with the 128-byte
    // swizzle and added by one TMA tensor reduction.
    bool ok = true;
    for (int it = 0; it < (DQ ? T : 0); ++it) {  // without the dQ path only the dV epilogue
      const int hq = hkv * G + (it0 + it) / nq;
      const int q0 = 64 * (qb0 + (it0 + it) % nq);
      const bool got = __all_sync(FULL, mbar_wait(dq_full(it & 1), (it >> 1) & 1, abort_flag, lim));
      uint32_t v[64];
      if (got) {
        tc_fence_after();
        const uint32_t dq_tm = tbase + lane_off + C::T_S + 64u * (it & 1);
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
        float* dst = p.dq_acc + (static_cast<long long>(b * p.Hq + hq) * p.Npad + q0) * D + r;
#pragma unroll
        for (int c = 0; c < 64; ++c) red_add_f32(dst + c * D, __uint_as_float(v[c]));
      } else {
        // The named barriers span the four warps, but a wait's outcome is only
        // warp-uniform: a warp that gives up records it in dq_fail and still arrives, after
        // which all four read the same flag and leave together.
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
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(rowp + ((u ^ (r & 7)) * 16)) = make_uint4(
                  v[32 * hh + 4 * u], v[32 * hh + 4 * u + 1], v[32 * hh + 4 * u + 2], v[32 * hh + 4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync_n(1, 128);
        if (r == 0) {
          const int bh = b * p.Hq + hq;
          tma_reduce_add_3d(&p.tm_dq, sbase + C::OFF_DQS, q0, 0, bh);
          tma_reduce_add_3d(&p.tm_dq, sbase + C::OFF_DQS + C::DQ_HALF, q0 + 32, 0, bh);
          bulk_commit_group();
        }
      }
    }
    if (C::DQ_TMA && r == 0) bulk_wait_group0();
    // ---- epilogue: dV -> 16-bit rows
    if (!ok) {
      wg_fail[2] = 1;
      fail();
    }
    if (!mbar_wait(acc_done, 0, abort_flag, lim)) {
      wg_fail[2] = 1;
      fail();
    }
    named_bar_sync_n(3, 128);
    if (wg_fail[2] == 0) {
      tc_fence_after();
      if (half >= 0) {
        bwd_add_partial<D>(tbase + lane_off + C::T_DV, smem + C::OFF_DO, &p.tm_kvpart, 2 * (unit - p.split_first) + 1,
                           3, r);
      } else {
        const int key = k0 + r;
        const long long krow = VARLEN ? static_cast<long long>(start_k) + key : static_cast<long long>(b) * N + key;
        bwd_write_tile<D, BF16, VARLEN>(tbase + lane_off + C::T_DV, 1.0f, smem + C::OFF_DO, &p.tm_dv,
                                        p.dv + (krow * p.Hkv + hkv) * D, key < len_k, 3, r, hkv, k0, b);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool DQ>
static cudaError_t launch_bwd_t(const BwdParams& args, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int sms = device_sm_count();
  BwdParams p = args;
  p.kv_part = nullptr;
  p.nsplit = 0;
  p.split_first = 0;
  const bool persistent = !VARLEN && bwd_persistent(p.N, CAUSAL);
  // Wave-tail split of the one-CTA-per-key-block grid (see BwdParams): when the grid's last
  // wave would occupy at most half of the SMs, its key blocks run as two half-walk CTAs
  // each, so that wave takes about half as long.  Needs room for the fp32 partials.
  if (!CAUSAL && !VARLEN && !persistent && sms > 0) {
    const long long units = static_cast<long long>((p.N + 127) / 128) * p.B * p.Hkv;
    const long long r = units % sms;
    const long long steps = static_cast<long long>(p.Hq / p.Hkv) * ((p.N + 63) / 64);
    const size_t bytes = static_cast<size_t>(r) * 2 * 128 * D * 4;
    if (r > 0 && 2 * r <= sms && steps >= 2 && p.part_space != nullptr && bytes <= p.part_bytes &&
        encode_dq_acc_map(&p.tm_kvpart, p.part_space, static_cast<int>(2 * r), D, 128)) {
      p.kv_part = p.part_space;
      p.nsplit = static_cast<int>(r);
      p.split_first = static_cast<int>(units - r);
    }
  }
  {
    // preprocess: LPR lanes per row, 8 rows per 256-thread block and step
    const long long rows = VARLEN ? static_cast<long long>(p.B) * p.Hq * p.Npad : static_cast<long long>(p.B) * p.N * p.Hq;
    const long long want = (rows * (D / 8) + 255) / 256;
    const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
    if (VARLEN)
      fa_bwd_preprocess_varlen<D, BF16><<<grid, 256, 0, stream>>>(p);
    else
      fa_bwd_preprocess<D, BF16><<<grid, 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // Deterministic pass: the dQ kernel reads only what the preprocess wrote, not the dK / dV
  // kernel's output, so it runs on the library's side stream, launched first (its CTAs are
  // the longer ones), while the dK / dV kernel runs on the caller's stream: each kernel's CTAs
  // then fill the SMs the other's last wave leaves idle.  The caller's stream waits for both.
  cudaStream_t side = nullptr;
  cudaEvent_t join = nullptr;
  cudaError_t e_side = cudaSuccess;
  if (!DQ && side_stream_fork(stream, &side, &join)) {
    e_side = launch_bwd_dq(p, D, BF16 ? FA_BF16 : FA_FP16, CAUSAL, side);
    const cudaError_t ej = cudaEventRecord(join, side);
    if (e_side == cudaSuccess) e_side = ej;
  }
  cudaError_t e_main = cudaSuccess;
  if (persistent) {
    e_main = launch_bwd_persistent(p, D, BF16, CAUSAL, DQ, stream);
  } else {
    auto kern = fa_bwd_main<D, BF16, CAUSAL, VARLEN, DQ>;
    e_main = prepare_launch_once<fa_bwd_main<D, BF16, CAUSAL, VARLEN, DQ>>(C::SMEM, C::THREADS, 128 * 80 + 256 * 160 + 128 * 112);
    const long long nk = VARLEN ? p.vl.max_k : p.N;
    const long long grid = ((nk + 127) / 128) * p.B * p.Hkv + p.nsplit;
    if (e_main == cudaSuccess && grid > 0) {
      kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(p);
      e_main = cudaGetLastError();
    }
    if (e_main == cudaSuccess && p.nsplit > 0) {
      // the split key blocks' dk / dv, before anything overwrites the partials (with the dQ
      // path they sit in dq, which the dQ convert below writes)
      const long long want = (static_cast<long long>(p.nsplit) * 2 * 128 * (D / 8) + 255) / 256;
      const int grid2 = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
      fa_bwd_split_convert<D, BF16><<<grid2, 256, 0, stream>>>(p);
      e_main = cudaGetLastError();
    }
  }
  if (side) {
    // join: the caller's stream goes on only once the side stream's dQ kernel is done
    const cudaError_t ew = cudaStreamWaitEvent(stream, join, 0);
    if (e_side != cudaSuccess) return e_side;
    if (e_main != cudaSuccess) return e_main;
    return ew;
  }
  if (e_main != cudaSuccess) return e_main;
  if (!DQ) return launch_bwd_dq(p, D, BF16 ? FA_BF16 : FA_FP16, CAUSAL, stream);
  if (BwdCfg<D>::DQ_TMA) {
    const long long grid = static_cast<long long>(p.B) * p.Hq * (VARLEN ? p.Npad / 64 : (p.N + 63) / 64);
    fa_bwd_dq_convert_t<D, BF16, VARLEN><<<static_cast<unsigned>(grid), 256, 0, stream>>>(p);
  } else {
    const long long threads = static_cast<long long>(p.B) * (VARLEN ? p.Npad : p.N) * p.Hq * (D / 8);
    const long long want = (threads + 255) / 256;
    const int grid = static_cast<int>(want < 16LL * sms ? (want > 0 ? want : 1) : 16LL * sms);
    fa_bwd_dq_convert<D, BF16, VARLEN><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

template <int D, bool BF16>
static cudaError_t launch_bwd_d(const BwdParams& p, bool causal, bool varlen, bool deterministic,
                                cudaStream_t stream) {
  if (varlen)
    return causal ? launch_bwd_t<D, BF16, true, true, true>(p, stream) : launch_bwd_t<D, BF16, false, true, true>(p, stream);
  if (deterministic)
    return causal ? launch_bwd_t<D, BF16, true, false, false>(p, stream)
                  : launch_bwd_t<D, BF16, false, false, false>(p, stream);
  return causal ? launch_bwd_t<D, BF16, true, false, true>(p, stream) : launch_bwd_t<D, BF16, false, false, true>(p, stream);
}

cudaError_t launch_bwd(const BwdParams& p, int d, fa_dtype dtype, bool causal, bool varlen, bool deterministic,
                       cudaStream_t stream) {
  const bool bf = dtype == FA_BF16;
  if (d == 128)
    return bf ? launch_bwd_d<128, true>(p, causal, varlen, deterministic, stream)
              : launch_bwd_d<128, false>(p, causal, varlen, deterministic, stream);
  return bf ? launch_bwd_d<64, true>(p, causal, varlen, deterministic, stream)
            : launch_bwd_d<64, false>(p, causal, varlen, deterministic, stream);
}

}  // namespace fa
