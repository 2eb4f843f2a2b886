// Device helpers shared by the backward's key-block kernels (one CTA per key block, and
// the persistent form for short sequences): 16-bit packing, the fp32 dQ reduction, the
// copy of V into tensor memory and the per-step P^T / dS^T arithmetic.
//
// The arithmetic is the textbook gradient of exact attention, recomputing P from the
// saved log-sum-exp ("FlashAttention-2: atención eficiente en GPU para contextos largos",
// section "Bloques pequeños, normalización global"):
//   P_ij  = exp(scale * q_i.k_j - lse_i)          (as exp2 with log2(e) folded in)
//   dS_ij = P_ij (dO_i.v_j - D_i)
#pragma once

#include "sm100_ptx.cuh"

#include <cuda_fp16.h>

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bw_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ float bw_unpack_lo(uint32_t v) {
  if (BF16) return __uint_as_float(v << 16);
  __half_raw hr;
  hr.x = static_cast<unsigned short>(v & 0xFFFFu);
  return __half2float(__half(hr));
}

template <bool BF16>
__device__ __forceinline__ float bw_unpack_hi(uint32_t v) {
  if (BF16) return __uint_as_float(v & 0xFFFF0000u);
  __half_raw hr;
  hr.x = static_cast<unsigned short>(v >> 16);
  return __half2float(__half(hr));
}

// global[p] += v, relaxed, without a result (a reduction, not a returning atomic)
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Row r of a V tile as the TMA loads it (64-column chunks of 128 rows x 128 B, 128-byte
// swizzle) -> TMEM lane r as 16-bit pairs from column `taddr` on (the A operand of
// dP^T = V dO^T).  The caller waits for the stores (tmem_wait_st) before announcing them.
template <int CHUNKS>
__device__ __forceinline__ void bwd_v_to_tmem(const uint8_t* v_tile, int r, uint32_t taddr) {
#pragma unroll
  for (int ch = 0; ch < CHUNKS; ++ch) {
    uint32_t kr[32];
    const uint8_t* rowp = v_tile + ch * (128 * 128) + r * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 q4 = *reinterpret_cast<const uint4*>(rowp + ((u ^ (r & 7)) * 16));
      kr[4 * u] = q4.x;
      kr[4 * u + 1] = q4.y;
      kr[4 * u + 2] = q4.z;
      kr[4 * u + 3] = q4.w;
    }
    tmem_st32(taddr + 32u * ch, kr);
  }
}

// P^T and dS^T of one key row (thread = key row) over 32 query columns of a step.
//   sv, dpv   S^T and dP^T of those columns (fp32 bit patterns, from TMEM)
//   nl4, nd4  per column -lse*log2(e) and -D (float4 groups in shared memory)
//   cmin      with a mask, columns below cmin see no key of this row (P = 0)
//   cl2x2     scale*log2(e), packed twice
//   rowp      with DQ, this row of the swizzled [128 keys x 64 queries] dS^T tile, of which
//             the caller's warpgroup `wg` writes 16-byte units [4 wg, 4 wg + 4)
//   pk, dsk   P^T and dS^T as 16-bit pairs (16 each), for TMEM
template <bool BF16, bool MASK, bool DQ>
__device__ __forceinline__ void bwd_p_ds(const uint32_t (&sv)[32], const uint32_t (&dpv)[32], const float4* nl4,
                                         const float4* nd4, int cmin, uint64_t cl2x2, uint8_t* rowp, int wg, int r,
                                         uint32_t (&pk)[16], uint32_t (&dsk)[16]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t* dk2 = dsk + 4 * g;
#pragma unroll
    for (int h4 = 0; h4 < 2; ++h4) {
      const int c4 = 2 * g + h4;
      const float4 L = nl4[c4], Dn = nd4[c4];
      // x = s * scale*log2(e) - lse*log2(e), two columns per instruction
      const uint64_t x01 = ffma2(f2pack(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), cl2x2,
                                 f2pack(L.x, L.y));
      const uint64_t x23 = ffma2(f2pack(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])),
                                 cl2x2, f2pack(L.z, L.w));
      float p0, p1, p2, p3;
      f2unpack(x01, p0, p1);
      f2unpack(x23, p2, p3);
      p0 = bw_ex2(p0);
      p1 = bw_ex2(p1);
      p2 = bw_ex2(p2);
      p3 = bw_ex2(p3);
      if (MASK) {
        if (4 * c4 + 0 < cmin) p0 = 0.f;
        if (4 * c4 + 1 < cmin) p1 = 0.f;
        if (4 * c4 + 2 < cmin) p2 = 0.f;
        if (4 * c4 + 3 < cmin) p3 = 0.f;
      }
      // dS = P * (dP - D)
      const uint64_t t01 = fadd2(f2pack(__uint_as_float(dpv[4 * c4]), __uint_as_float(dpv[4 * c4 + 1])),
                                 f2pack(Dn.x, Dn.y));
      const uint64_t t23 = fadd2(f2pack(__uint_as_float(dpv[4 * c4 + 2]), __uint_as_float(dpv[4 * c4 + 3])),
                                 f2pack(Dn.z, Dn.w));
      float d0, d1, d2, d3;
      f2unpack(fmul2(f2pack(p0, p1), t01), d0, d1);
      f2unpack(fmul2(f2pack(p2, p3), t23), d2, d3);
      pk[2 * c4] = pack_half2<BF16>(p0, p1);
      pk[2 * c4 + 1] = pack_half2<BF16>(p2, p3);
      dk2[2 * h4] = pack_half2<BF16>(d0, d1);
      dk2[2 * h4 + 1] = pack_half2<BF16>(d2, d3);
    }
    if (DQ)  // the shared-memory copy of dS^T feeds only the dQ^T product
      *reinterpret_cast<uint4*>(rowp + (((4 * wg + g) ^ (r & 7)) * 16)) = make_uint4(dk2[0], dk2[1], dk2[2], dk2[3]);
  }
}

}  // namespace fa
