// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Device error word bits (set by kernels whose bounded waits ran out).
constexpr unsigned kDevErrTimeout = 1u;

// Bounded waits give up after this long (ns); a pipeline stage normally waits
// microseconds, so only a broken pipeline gets near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 4-D maps over [B, N, H, d] (d innermost)
  float* lse;                          // [B, Hq, N]
  unsigned* err;                       // device error word
  int B, Hq, Hkv, N;
  float scale_log2;                    // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
};

// Encodes a 4-D tensor map over a [B, N, H, d] 16-bit tensor, box = {64, 1, rows, 1},
// 128-byte swizzle.  Returns false if the driver rejects it.
bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows,
                     fa_dtype dtype);

unsigned* device_error_word();  // address of this device's error word (device memory)

cudaError_t launch_fwd(const FwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);

}  // namespace fa
