// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Device error word bits: a bounded wait ran out / a launch found its shared-memory
// base misaligned (did no work).
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrLayout = 2u;
// A variable-length launch found a sequence whose offsets or length contradict the
// sizes it was given (it wrote nothing for that sequence).
constexpr unsigned kDevErrSeqlens = 4u;

// Bounded waits give up after this long (ns); a pipeline stage normally waits
// microseconds, so only a broken pipeline gets near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Variable-length batches: sequence b owns rows [cu[b], cu[b+1]) of the packed
// [total, H, d] tensors, of which the first len_b are real (len_b = used[b] when `used`
// is given, else cu[b+1] - cu[b]).  Device pointers; all null for fixed-length calls.
struct Seqlens {
  const int* cu_q;
  const int* cu_k;
  const int* used_q;
  const int* used_k;
  int total_q, total_k;  // rows of the packed tensors
  int max_q, max_k;      // upper bounds on len_b (size the grid)
};

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;  // fixed: 4-D maps over [B, N, H, d]; varlen: 3-D over [total, H, d]
  float* lse;                          // fixed: [B, Hq, N]; varlen: [Hq, total_q]
  uint16_t* o;                         // varlen: rows of tiles that end past their sequence
  unsigned* err;                       // device error word
  int B, Hq, Hkv, N;
  float scale_log2;                    // scale * log2(e)
  float scale;
  uint64_t wait_limit_ns;
  Seqlens vl;
};

// Encodes a 4-D tensor map over a [B, N, H, d] 16-bit tensor, box = {64, 1, rows, 1},
// 128-byte swizzle.  Returns false if the driver rejects it.
bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows,
                     fa_dtype dtype);
// 3-D map over a packed [total, H, d] 16-bit tensor, box = {64, 1, rows}, 128-byte swizzle.
// 4-D map over a [B, N, H, d] 16-bit tensor with box = {64, box_h, box_rows, 1}.
bool encode_bshd_box_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_h, int box_rows,
                         fa_dtype dtype);
bool encode_thd_map(CUtensorMap* map, const void* base, int total, int H, int d, int box_rows, fa_dtype dtype);

struct BwdParams {
  CUtensorMap tm_q, tm_do;  // [B, N, Hq, d], box rows 64
  CUtensorMap tm_k, tm_v;   // [B, N, Hkv, d], box rows 128
  CUtensorMap tm_dk, tm_dv; // fixed length: outputs [B, N, Hkv, d] (TMA stores), box rows 128, or 32 for the
                            // persistent kernel (each warp stores its own 32 key rows)
  CUtensorMap tm_dq;        // d=64: fp32 dQ accumulator [B*Hq, d, Npad], box {32, d, 1}, 128-byte swizzle
  const uint16_t* o;        // [B, N, Hq, d] (preprocess)
  const uint16_t* dout;     // [B, N, Hq, d] (preprocess)
  const float* lse;         // [B, Hq, N]
  uint16_t* dq;             // [B, N, Hq, d]
  uint16_t* dk;             // [B, N, Hkv, d]
  uint16_t* dv;             // [B, N, Hkv, d]
  float* dq_acc;            // workspace: fp32, [B*Hq, Npad, d] at d=128, [B*Hq, d, Npad] at d=64
  float* dvec;              // workspace: -D = -rowsum(dO*O), [B*Hq, Npad] (0 past N)
  float* l2vec;             // workspace: -lse * log2(e), [B*Hq, Npad] (-inf past N)
  unsigned* err;
  int B, Hq, Hkv, N, Npad;  // varlen: N unused, Npad = max_q rounded up to 64 (at least 64)
  float scale, scale_log2;
  uint64_t wait_limit_ns;
  Seqlens vl;  // varlen: packed layouts ([total, H, d] tensors, lse [Hq, total_q])
  // Wave-tail split (fixed length, non-causal, one CTA per key block): the last nsplit key
  // blocks of the grid run as two CTAs each, one per half of the query walk, which add
  // their fp32 dK / dV into kv_part [nsplit][2 (dK, dV)][128][d] (zeroed by the
  // preprocess; TMA map tm_kvpart, 3-D {d, 128, 2 nsplit}, box {32, 128, 1}), and
  // fa_bwd_split_convert writes those blocks' dk / dv.  Key block u >= split_first runs
  // as CTAs split_first + 2 (u - split_first) + h.  part_space / part_bytes: memory the
  // call may use for kv_part (fa_bwd: the dq output, written only at the end;
  // fa_bwd_deterministic: the unused fp32 dQ accumulator); null / 0 where the split is off.
  CUtensorMap tm_kvpart;
  float* kv_part;
  int split_first, nsplit;
  float* part_space;
  size_t part_bytes;
};

// Decode-shaped forward with split keys.
struct DecParams {
  CUtensorMap tm_q;        // 4-D over q [B, Nq, Hq, d], box {64, G, Nq, 1}: the group's rows
  CUtensorMap tm_k, tm_v;  // 4-D over the caches [B, Nmax, Hkv, d] (paged: [num_pages, 128, Hkv, d]),
                           // box {64, 1, 128, 1}
  const int* seqlens_k;    // [B] keys in the cache of each sequence (device)
  const int* block_table;  // paged caches: [B, max_pages] page of each 128-key block (device); else null
  int max_pages, num_pages;
  uint16_t* o;             // [B, Nq, Hq, d]
  float* lse;              // [B, Hq, Nq]
  float* opart;            // splits > 1: [B*Hkv*S, M, d] normalised partial outputs (fp32)
  float* lpart;            // splits > 1: [B*Hkv*S, M] partial log-sum-exp
  unsigned* err;
  int B, Hq, Hkv, Nq, Nmax;
  int G, M;                // G = Hq / Hkv, M = G * Nq packed rows (<= 128)
  int S, cps;              // splits, key blocks of 128 per split
  float scale, scale_log2;
  uint64_t wait_limit_ns;
};
cudaError_t launch_decode(const DecParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);

// FP8 (E4M3) forward, head dimension 128.
struct Fp8Params {
  CUtensorMap tm_q, tm_k;  // 4-D over E4M3 [B, N, H, 128], box {128, 1, 128, 1}, 128-byte swizzle
  CUtensorMap tm_vt;       // 3-D over V^T [B*Hkv, 128, Npad] (keys contiguous), box {128, 128, 1}
  const uint8_t* v;        // [B, N, Hkv, 128] E4M3 (input of the transpose)
  uint8_t* vt;             // workspace: V^T, zero past N
  uint16_t* o;             // [B, N, Hq, 128] bf16
  float* lse;              // [B, Hq, N]
  unsigned* err;
  int B, Hq, Hkv, N, Npad;  // Npad = N rounded up to 128
  float score_log2;         // scale * q_descale * k_descale * log2(e)
  float score_scale;        // scale * q_descale * k_descale
  float out_scale;          // v_descale (P and its row sum both carry a 2^8 pre-scale)
  uint64_t wait_limit_ns;
  // per-block descales (fa_fwd_fp8_blockscaled; null for one descale per tensor): one fp32
  // per 128-row block of each head, q_bs [B, Hq, nb], k_bs and v_bs [B, Hkv, nb],
  // nb = ceil(N / 128)
  const float* q_bs;
  const float* k_bs;
  const float* v_bs;
  int nb;
  float scale_log2;  // scale * log2(e)
};
cudaError_t launch_fwd_fp8(const Fp8Params& p, bool causal, cudaStream_t stream);
// 4-D map over an 8-bit [B, N, H, d] tensor, box {d, 1, rows, 1} (d = 128 bytes).
bool encode_bshd_u8_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows);
// 3-D map over an 8-bit [BH, d, Npad] tensor, box {128, d, 1}.
bool encode_vt_u8_map(CUtensorMap* map, const void* base, int BH, int d, int Npad);

// Workspace layout for the backward pass (all offsets 256-byte aligned).
struct BwdWorkspace {
  size_t dq_acc_off, dvec_off, l2vec_off, total;
};
BwdWorkspace bwd_workspace_layout(int B, int Hq, int N, int d);


// 3-D map over the fp32 dQ accumulator [BH, d, Npad] (queries contiguous), box {32, d, 1},
// 128-byte swizzle: the target of the d=64 backward's tensor reductions.
bool encode_dq_acc_map(CUtensorMap* map, const float* base, int BH, int Npad, int d);

unsigned* device_error_word();  // address of this device's error word (device memory)

// First-launch preparation of kernel `Kern` on the current device, done once per device:
//  - raises its dynamic shared-memory limit to `smem_bytes` (the attribute belongs to the
//    function on the device and stays set, so repeating it per launch only costs time);
//  - checks its register split: a kernel whose warpgroups rebalance registers with
//    setmaxnreg needs `split_regs` registers in total (threads x registers of every role
//    after the rebalancing), and setmaxnreg.inc draws only on the block's own launch
//    allocation (threads x the compiled register count, in steps of 8 per thread).  A
//    split above that would make setmaxnreg.inc wait forever, so the launch is refused.
// (Devices 64 and up repeat the preparation on every call.)
template <auto Kern>
cudaError_t prepare_launch_once(int smem_bytes, int threads, int split_regs) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  if (split_regs > 0) {
    cudaFuncAttributes attr{};
    e = cudaFuncGetAttributes(&attr, Kern);
    if (e != cudaSuccess) return e;
    const long long per_thread = (static_cast<long long>(attr.numRegs) + 7) / 8 * 8;
    if (per_thread * threads < split_regs) return cudaErrorInvalidConfiguration;
  }
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Streaming-multiprocessor count of the current device (looked up once per device).
int device_sm_count();
// Fork for two independent launches: after this call, work enqueued on *side starts only
// once the work enqueued on `stream` so far has finished; the caller then records *join on
// *side and makes `stream` wait for it.  The side stream (non-blocking) and a ring of
// kSideEvents event pairs are created once per device; calls that overlap in time get
// different pairs unless kSideEvents calls separate them.  Returns false (nothing enqueued)
// if the device's side stream or events cannot be had; the caller then stays on `stream`.
constexpr int kSideEvents = 64;
bool side_stream_fork(cudaStream_t stream, cudaStream_t* side, cudaEvent_t* join);

cudaError_t launch_fwd(const FwdParams& p, int d, fa_dtype dtype, bool causal, bool varlen, cudaStream_t stream);
// Persistent forward (fixed length): one CTA per SM takes units from a counter pair
// {next, done} in device memory.  Each launch takes the next pair of a ring of
// kSchedSlots per device (round robin over all launches of the process); the launch's
// last CTA puts the pair back to {0, 0}.  Two launches that use one pair at the same time
// (kSchedSlots launches apart, still running together) would share its units.
constexpr int kSchedSlots = 256;
// fa_fwd runs the persistent kernel up to these sequence lengths (few key blocks per unit,
// where a unit's start and finish cost as much as its blocks) and one CTA per unit above;
// both limits are where the persistent kernel stopped measuring faster
constexpr int kPersistentMaxN = 512;
constexpr int kPersistentMaxNCausal = 1024;
constexpr int kMaxSchedDevices = 64;
unsigned* scheduler_slot();  // nullptr if the device's ring cannot be found
cudaError_t launch_fwd_persistent(const FwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);
// deterministic: dK/dV from the key-block kernel without its dQ path, then dQ from the
// query-tile kernel (fa_bwd_dq.cu) in a fixed summation order; p.dq_acc must be null.
cudaError_t launch_bwd(const BwdParams& p, int d, fa_dtype dtype, bool causal, bool varlen, bool deterministic,
                       cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdParams& p, int d, fa_dtype dtype, bool causal, cudaStream_t stream);
// Persistent form of the key-block backward kernel (fixed length; fa_bwd_persist.cu): one
// CTA per SM takes (batch, key/value head, key block) units from a counter pair of the
// ring above.  dq = false leaves out the dQ path, as the deterministic pass wants.  The
// backward uses it up to these sequence lengths and one CTA per key block above.
constexpr int kPersistentBwdMaxN = 512;
constexpr int kPersistentBwdMaxNCausal = 512;
inline bool bwd_persistent(int N, bool causal) {
  return N <= (causal ? kPersistentBwdMaxNCausal : kPersistentBwdMaxN);
}
cudaError_t launch_bwd_persistent(const BwdParams& p, int d, bool bf16, bool causal, bool dq, cudaStream_t stream);

// Geometry of sequence b of a variable-length launch; false if its offsets or length
// contradict the launch's sizes.
__device__ __forceinline__ bool seq_span(const Seqlens& vl, int b, int& start_q, int& len_q, int& start_k,
                                         int& len_k) {
  const int sq = vl.cu_q[b], eq = vl.cu_q[b + 1], sk = vl.cu_k[b], ek = vl.cu_k[b + 1];
  const int lq = vl.used_q ? vl.used_q[b] : eq - sq;
  const int lk = vl.used_k ? vl.used_k[b] : ek - sk;
  start_q = sq;
  len_q = lq;
  start_k = sk;
  len_k = lk;
  return sq >= 0 && eq >= sq && eq <= vl.total_q && lq >= 0 && lq <= eq - sq && lq <= vl.max_q && sk >= 0 &&
         ek >= sk && ek <= vl.total_k && lk >= 0 && lk <= ek - sk && lk <= vl.max_k;
}

}  // namespace fa
