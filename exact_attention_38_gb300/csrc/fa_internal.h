// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Device error word bits: a bounded wait ran out / a launch found its shared-memory
// base misaligned (did no work).
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrLayout = 2u;

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

struct BwdParams {
  CUtensorMap tm_q, tm_do;  // [B, N, Hq, d], box rows 64
  CUtensorMap tm_k, tm_v;   // [B, N, Hkv, d], box rows 128
  CUtensorMap tm_dq;        // fp32 dQ accumulator [B*Hq, d, Npad], box {32, d, 1}, 128-byte swizzle
  const uint16_t* o;        // [B, N, Hq, d] (preprocess)
  const uint16_t* dout;     // [B, N, Hq, d] (preprocess)
  const float* lse;         // [B, Hq, N]
  uint16_t* dq;             // [B, N, Hq, d]
  uint16_t* dk;             // [B, N, Hkv, d]
  uint16_t* dv;             // [B, N, Hkv, d]
  float* dq_acc;            // workspace: fp32 [B*Hq, d, Npad] (queries contiguous)
  float* dvec;              // workspace: -D = -rowsum(dO*O), [B*Hq, Npad] (0 past N)
  float* l2vec;             // workspace: -lse * log2(e), [B*Hq, Npad] (-inf past N)
  unsigned* err;
  int B, Hq, Hkv, N, Npad;
  float scale, scale_log2;
  uint64_t wait_limit_ns;
};

// Workspace layout for the backward pass (all offsets 256-byte aligned).
struct BwdWorkspace {
  size_t dq_acc_off, dvec_off, l2vec_off, total;
};
BwdWorkspace bwd_workspace_layout(int B, int Hq, int N, int d);

// 3-D map over the fp32 dQ accumulator [B*Hq, d, Npad], box = {32, d, 1}, 128-byte swizzle.
bool encode_dq_acc_map(CUtensorMap* map, const float* base, int BH, int Npad, int d);

unsigned* device_error_word();  // address of this device's error word (device memory)

cudaError_t launch_fwd(const FwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);
cudaError_t launch_bwd(const BwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);

}  // namespace fa
