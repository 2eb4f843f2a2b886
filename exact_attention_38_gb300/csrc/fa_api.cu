// C ABI of libfa.so: argument validation, tensor-map encoding, launches.
// Every argument check happens before the first CUDA call, so a bad call returns
// an error code without touching the device (and works on a host without a GPU).
#include "fa_decode_policy.h"
#include "fa_internal.h"
#include "fa_math.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

namespace fa {

__device__ unsigned g_fa_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_err_ptr[kMaxDevices];
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  PFN_cuTensorMapEncodeTiled_v12000 f = g_encode.load(std::memory_order_acquire);
  if (f) return f;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return nullptr;
  f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  g_encode.store(f, std::memory_order_release);
  return f;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by forward and backward.
fa_status check_sizes(int B, int Hq, int Hkv, int N, int d, float scale, int dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return FA_ERR_INVALID;
  if (Hq % Hkv != 0) return FA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (N > (1 << 20)) return FA_ERR_UNSUPPORTED;
  // element counts must fit the tensor maps and 2^31 CTAs
  const long long rows = static_cast<long long>(B) * N;
  if (rows * Hq * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  const long long tiles = static_cast<long long>(B) * Hq * ((N + 255) / 256);
  if (tiles >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Shape checks of the variable-length entry points (the per-sequence offsets live in
// device memory and are checked by the kernels).
fa_status check_varlen(int B, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k, int d, float scale,
                       int dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || total_q < 0 || total_k < 0 || max_q < 0 || max_k < 0)
    return FA_ERR_INVALID;
  if (Hq % Hkv != 0) return FA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (max_q > (1 << 20) || max_k > (1 << 20) || B > (1 << 20)) return FA_ERR_UNSUPPORTED;
  const long long tq = static_cast<long long>(total_q) * Hq * d * 2, tk = static_cast<long long>(total_k) * Hkv * d * 2;
  if (tq >= (1LL << 40) || tk >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  const long long tiles = static_cast<long long>(B) * Hq * ((max_q + 255) / 256);
  const long long kblocks = static_cast<long long>(B) * Hkv * ((max_k + 127) / 128);
  if (tiles >= (1LL << 31) || kblocks >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

bool aligned4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Split count of the decode pass: as many splits as fit one wave of CTA slots on a
// 152-SM part (304 at two CTAs per SM, or 152 with the deep K/V ring of
// decode_deep_ring; a fixed target, so the workspace size does not depend on the
// device; measured best on GB300 against 2-4x more CTAs), never more splits than key
// blocks; `want` > 0 overrides the target.
struct DecodeSplit {
  int S, cps;
};
DecodeSplit decode_split(int B, int Hkv, int Nmax, int d, int want) {
  const int nkb = (Nmax + 127) / 128;
  const long long units = static_cast<long long>(B) * Hkv;
  long long S = want > 0 ? want : decode_cta_slots(d, units) / units;
  if (S > nkb) S = nkb;
  if (S < 1) S = 1;
  const int cps = static_cast<int>((nkb + S - 1) / S);
  return {static_cast<int>((nkb + cps - 1) / cps), cps};
}

fa_status check_decode(int B, int Hq, int Hkv, int Nq, int Nmax, int d, float scale, int dtype, int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nmax < 1 || d < 1 || num_splits < 0) return FA_ERR_INVALID;
  if (Hq % Hkv != 0) return FA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((Hq / Hkv) * Nq > 128) return FA_ERR_UNSUPPORTED;  // the group's rows fill one 128-row tile
  if (Nmax > (1 << 24)) return FA_ERR_UNSUPPORTED;
  const long long kv = static_cast<long long>(B) * Nmax * Hkv * d * 2;
  if (kv >= (1LL << 40) || static_cast<long long>(B) * Nq * Hq * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hkv * decode_split(B, Hkv, Nmax, d, num_splits).S >= (1LL << 31))
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

struct DecodeWorkspace {
  size_t opart_off, lpart_off, total;
};
DecodeWorkspace decode_workspace_layout(int B, int Hq, int Hkv, int Nq, int Nmax, int d, int num_splits) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const DecodeSplit sp = decode_split(B, Hkv, Nmax, d, num_splits);
  DecodeWorkspace w{};
  if (sp.S == 1) return w;
  const size_t rows = static_cast<size_t>(B) * Hkv * sp.S * (Hq / Hkv) * Nq;
  w.opart_off = 0;
  w.lpart_off = up(rows * d * 4);
  w.total = w.lpart_off + up(rows * 4);
  return w;
}

}  // namespace

BwdWorkspace bwd_workspace_layout(int B, int Hq, int N, int d) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t npad = (static_cast<size_t>(N) + 63) / 64 * 64;
  BwdWorkspace w{};
  w.dq_acc_off = 0;
  w.dvec_off = up(static_cast<size_t>(B) * Hq * d * npad * 4);
  w.l2vec_off = w.dvec_off + up(static_cast<size_t>(B) * Hq * npad * 4);
  w.total = w.l2vec_off + up(static_cast<size_t>(B) * Hq * npad * 4);
  return w;
}

unsigned* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_fa_error_word) != cudaSuccess) return nullptr;
  p = static_cast<unsigned*>(addr);
  g_err_ptr[dev].store(p, std::memory_order_release);
  return p;
}

bool side_stream_fork(cudaStream_t stream, cudaStream_t* side, cudaEvent_t* join) {
  struct Side {
    cudaStream_t stream;
    cudaEvent_t ev[kSideEvents][2];
  };
  static std::atomic<Side*> state[kMaxDevices];
  static std::mutex mu;
  static std::atomic<unsigned> next{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  Side* st = state[dev].load(std::memory_order_acquire);
  if (!st) {
    std::lock_guard<std::mutex> lock(mu);
    st = state[dev].load(std::memory_order_acquire);
    if (!st) {
      Side* n = new Side{};
      bool ok = cudaStreamCreateWithFlags(&n->stream, cudaStreamNonBlocking) == cudaSuccess;
      for (int i = 0; i < kSideEvents && ok; ++i)
        for (int j = 0; j < 2 && ok; ++j)
          ok = cudaEventCreateWithFlags(&n->ev[i][j], cudaEventDisableTiming) == cudaSuccess;
      if (!ok) {
        cudaGetLastError();
        return false;  // (the partly created set is left in place; this happens at most once)
      }
      state[dev].store(n, std::memory_order_release);
      st = n;
    }
  }
  const unsigned i = next.fetch_add(1u, std::memory_order_relaxed) % kSideEvents;
  if (cudaEventRecord(st->ev[i][0], stream) != cudaSuccess || cudaStreamWaitEvent(st->stream, st->ev[i][0], 0) != cudaSuccess)
    return false;
  *side = st->stream;
  *join = st->ev[i][1];
  return true;
}

int device_sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 148;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(sms, std::memory_order_release);
  return sms;
}

bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows,
                     fa_dtype dtype) {
  return encode_bshd_box_map(map, base, B, N, H, d, 1, box_rows, dtype);
}

bool encode_bshd_box_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_h, int box_rows,
                         fa_dtype dtype) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t es = 2;
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(H) * d * es,
                                 static_cast<cuuint64_t>(N) * H * d * es};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r =
      enc(map, dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_thd_map(CUtensorMap* map, const void* base, int total, int H, int d, int box_rows, fa_dtype dtype) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  // an empty packed tensor is never read (every sequence has length 0); the map still
  // needs one row to be encodable
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(total > 0 ? total : 1)};
  const cuuint64_t es = 2;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(H) * d * es};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(map, dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_bshd_u8_map(CUtensorMap* map, const void* base, int B, int N, int H, int d, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d,
                                 static_cast<cuuint64_t>(N) * H * d};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_vt_u8_map(CUtensorMap* map, const void* base, int BH, int d, int Npad) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(Npad), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Npad), static_cast<cuuint64_t>(d) * Npad};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(d), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_dq_acc_map(CUtensorMap* map, const float* base, int BH, int Npad, int d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(Npad), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Npad) * 4, static_cast<cuuint64_t>(d) * Npad * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(d), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Waits on an mbarrier that no thread ever arrives on, through the same bounded wait the
// attention kernels use; the wait gives up after `limit_ns` and records the timeout.
__global__ void fa_selftest_wait_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(smem_u32(&bar), 0, nullptr, limit_ns);
  if (!ok && threadIdx.x == 0) atomicOr(err, kDevErrTimeout);
}

// Evaluates both exponential forms the softmax kernels use, element by element.
__global__ void fa_selftest_exp2_kernel(const float* x, float* y_poly, float* y_mufu, int n) {
  const long long i = 2LL * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const bool two = i + 1 < n;
  const float x0 = x[i], x1 = two ? x[i + 1] : 0.f;
  float p0, p1;
  f2unpack(ex2_poly2(f2pack(x0, x1)), p0, p1);
  y_poly[i] = p0;
  y_mufu[i] = ex2_mufu(x0);
  if (two) {
    y_poly[i + 1] = p1;
    y_mufu[i + 1] = ex2_mufu(x1);
  }
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: valid but unsupported size or head dimension";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel's bounded wait ran out";
  }
  return "unknown fa_status";
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                 int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID;
  const fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  FwdParams p{};
  if (!encode_bshd_map(&p.tm_q, q, B, N, Hq, d, 128, dtype) || !encode_bshd_map(&p.tm_k, k, B, N, Hkv, d, 128, dtype) ||
      !encode_bshd_map(&p.tm_v, v, B, N, Hkv, d, 128, dtype) || !encode_bshd_map(&p.tm_o, o, B, N, Hq, d, 128, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  p.lse = lse;
  p.o = static_cast<uint16_t*>(o);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool persistent = N <= (causal ? kPersistentMaxNCausal : kPersistentMaxN);
  const cudaError_t e = persistent ? launch_fwd_persistent(p, d, dtype, causal != 0, s)
                                   : launch_fwd(p, d, dtype, causal != 0, false, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, const int* seqused_q, const int* seqused_k, int B, int Hq, int Hkv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, int causal, float scale,
                        fa_dtype dtype, fa_stream_t stream) {
  if (!aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k)) return FA_ERR_INVALID;
  if ((seqused_q && !aligned4(seqused_q)) || (seqused_k && !aligned4(seqused_k))) return FA_ERR_INVALID;
  const fa_status st =
      check_varlen(B, Hq, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  if (total_q == 0 || max_seqlen_q == 0) return FA_OK;  // no query row to write
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID;
  if (total_k > 0 && (!aligned16(k) || !aligned16(v))) return FA_ERR_INVALID;
  // with no key row at all the key/value maps are never read; they are encoded over q
  const void* kb = total_k > 0 ? k : q;
  const void* vb = total_k > 0 ? v : q;
  FwdParams p{};
  if (!encode_thd_map(&p.tm_q, q, total_q, Hq, d, 128, dtype) || !encode_thd_map(&p.tm_k, kb, total_k, Hkv, d, 128, dtype) ||
      !encode_thd_map(&p.tm_v, vb, total_k, Hkv, d, 128, dtype) || !encode_thd_map(&p.tm_o, o, total_q, Hq, d, 128, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  p.lse = lse;
  p.o = static_cast<uint16_t*>(o);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  p.vl = Seqlens{cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k, total_q, total_k, max_seqlen_q, max_seqlen_k};
  const cudaError_t e = launch_fwd(p, d, dtype, causal != 0, true, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d) {
  if (check_sizes(B, Hq, Hkv, N, d, 1.0f, FA_BF16) != FA_OK) return 0;
  return bwd_workspace_layout(B, Hq, N, d).total;
}

}  // extern "C"

namespace {
fa_status bwd_fixed(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                    fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream,
                    bool deterministic) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  const fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  const BwdWorkspace ws = bwd_workspace_layout(B, Hq, N, d);
  if (workspace_bytes < ws.total) return FA_ERR_INVALID;
  BwdParams p{};
  const int out_rows = bwd_persistent(N, causal != 0) ? 32 : 128;
  if (!encode_bshd_map(&p.tm_q, q, B, N, Hq, d, 64, dtype) || !encode_bshd_map(&p.tm_do, dout, B, N, Hq, d, 64, dtype) ||
      !encode_bshd_map(&p.tm_k, k, B, N, Hkv, d, 128, dtype) || !encode_bshd_map(&p.tm_v, v, B, N, Hkv, d, 128, dtype) ||
      !encode_bshd_map(&p.tm_dk, dk, B, N, Hkv, d, out_rows, dtype) ||
      !encode_bshd_map(&p.tm_dv, dv, B, N, Hkv, d, out_rows, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.dq_acc = deterministic ? nullptr : reinterpret_cast<float*>(w + ws.dq_acc_off);
  p.dvec = reinterpret_cast<float*>(w + ws.dvec_off);
  p.l2vec = reinterpret_cast<float*>(w + ws.l2vec_off);
  if (!deterministic && d == 64 && !encode_dq_acc_map(&p.tm_dq, p.dq_acc, B * Hq, (N + 63) / 64 * 64, d))
    return FA_ERR_CUDA;
  // room for the wave-tail split's fp32 dK / dV partials (see BwdParams): fa_bwd keeps them
  // in dq, which it otherwise writes only at the end, so not when dq's memory overlaps an
  // input of the pass (the split would overwrite it before it is read)
  const size_t q_bytes = static_cast<size_t>(B) * N * Hq * d * 2, kv_bytes = static_cast<size_t>(B) * N * Hkv * d * 2;
  auto overlaps = [&](const void* a, size_t na) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(dq);
    return x < y + q_bytes && y < x + na;
  };
  const bool dq_clear = !overlaps(q, q_bytes) && !overlaps(k, kv_bytes) && !overlaps(v, kv_bytes) &&
                        !overlaps(o, q_bytes) && !overlaps(dout, q_bytes) &&
                        !overlaps(lse, static_cast<size_t>(B) * Hq * N * 4);
  p.part_space = deterministic ? reinterpret_cast<float*>(w + ws.dq_acc_off)
                 : dq_clear    ? static_cast<float*>(dq)
                               : nullptr;
  p.part_bytes = deterministic ? ws.dvec_off - ws.dq_acc_off : dq_clear ? q_bytes : 0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.Npad = (N + 63) / 64 * 64;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  const cudaError_t e =
      launch_bwd(p, d, dtype, causal != 0, false, deterministic, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

extern "C" {

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_fixed(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, false);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                               int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                               fa_stream_t stream) {
  return bwd_fixed(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, true);
}


static int varlen_npad(int max_q) { return max_q > 0 ? (max_q + 63) / 64 * 64 : 64; }

size_t fa_bwd_varlen_workspace_size(int B, int Hq, int max_seqlen_q, int d) {
  if (check_varlen(B, Hq, 1, 0, 0, max_seqlen_q, 0, d, 1.0f, FA_BF16) != FA_OK) return 0;
  return bwd_workspace_layout(B, Hq, varlen_npad(max_seqlen_q), d).total;
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, const int* seqused_q, const int* seqused_k, int B, int Hq, int Hkv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, int causal, float scale,
                        fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k)) return FA_ERR_INVALID;
  if ((seqused_q && !aligned4(seqused_q)) || (seqused_k && !aligned4(seqused_k))) return FA_ERR_INVALID;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  const fa_status st =
      check_varlen(B, Hq, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d, scale, static_cast<int>(dtype));
  if (st != FA_OK) return st;
  const int npad = varlen_npad(max_seqlen_q);
  const BwdWorkspace ws = bwd_workspace_layout(B, Hq, npad, d);
  if (workspace_bytes < ws.total) return FA_ERR_INVALID;
  if (total_q == 0 && total_k == 0) return FA_OK;  // nothing to write
  if (total_q > 0 && (!aligned16(q) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) || !aligned16(dq)))
    return FA_ERR_INVALID;
  if (total_k > 0 && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))) return FA_ERR_INVALID;
  // an empty side is never read (every sequence has length 0 there); its maps are
  // encoded over the other side's tensors
  const void* qb = total_q > 0 ? q : k;
  const void* dob = total_q > 0 ? dout : k;
  const void* kb = total_k > 0 ? k : q;
  const void* vb = total_k > 0 ? v : q;
  BwdParams p{};
  if (!encode_thd_map(&p.tm_q, qb, total_q, Hq, d, 64, dtype) || !encode_thd_map(&p.tm_do, dob, total_q, Hq, d, 64, dtype) ||
      !encode_thd_map(&p.tm_k, kb, total_k, Hkv, d, 128, dtype) || !encode_thd_map(&p.tm_v, vb, total_k, Hkv, d, 128, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  p.o = static_cast<const uint16_t*>(o);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.dq_acc = reinterpret_cast<float*>(w + ws.dq_acc_off);
  p.dvec = reinterpret_cast<float*>(w + ws.dvec_off);
  p.l2vec = reinterpret_cast<float*>(w + ws.l2vec_off);
  if (d == 64 && !encode_dq_acc_map(&p.tm_dq, p.dq_acc, B * Hq, npad, d)) return FA_ERR_CUDA;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = 0;
  p.Npad = npad;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  p.vl = Seqlens{cu_seqlens_q, cu_seqlens_k, seqused_q, seqused_k, total_q, total_k, max_seqlen_q, max_seqlen_k};
  const cudaError_t e = launch_bwd(p, d, dtype, causal != 0, true, false, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int Nmax, int d, int num_splits) {
  if (check_decode(B, Hq, Hkv, Nq, Nmax, d, 1.0f, FA_BF16, num_splits) != FA_OK) return 0;
  return decode_workspace_layout(B, Hq, Hkv, Nq, Nmax, d, num_splits).total;
}

int fa_decode_num_splits(int B, int Hq, int Hkv, int Nq, int Nmax, int d, int num_splits) {
  if (check_decode(B, Hq, Hkv, Nq, Nmax, d, 1.0f, FA_BF16, num_splits) != FA_OK) return 0;
  return decode_split(B, Hkv, Nmax, d, num_splits).S;
}

fa_status fa_fwd_decode(const void* q, const void* k_cache, const void* v_cache, const int* cache_seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int Nq, int Nmax, int d, int causal, float scale,
                        int num_splits, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                        fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID;
  if (!aligned4(cache_seqlens)) return FA_ERR_INVALID;
  const fa_status st = check_decode(B, Hq, Hkv, Nq, Nmax, d, scale, static_cast<int>(dtype), num_splits);
  if (st != FA_OK) return st;
  const DecodeSplit sp = decode_split(B, Hkv, Nmax, d, num_splits);
  const DecodeWorkspace ws = decode_workspace_layout(B, Hq, Hkv, Nq, Nmax, d, num_splits);
  if (ws.total > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                       workspace_bytes < ws.total))
    return FA_ERR_INVALID;
  const int G = Hq / Hkv;
  DecParams p{};
  if (!encode_bshd_box_map(&p.tm_q, q, B, Nq, Hq, d, G, Nq, dtype) ||
      !encode_bshd_map(&p.tm_k, k_cache, B, Nmax, Hkv, d, 128, dtype) ||
      !encode_bshd_map(&p.tm_v, v_cache, B, Nmax, Hkv, d, 128, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  p.seqlens_k = cache_seqlens;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.opart = ws.total ? reinterpret_cast<float*>(w + ws.opart_off) : nullptr;
  p.lpart = ws.total ? reinterpret_cast<float*>(w + ws.lpart_off) : nullptr;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nmax = Nmax;
  p.G = G;
  p.M = G * Nq;
  p.S = sp.S;
  p.cps = sp.cps;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  const cudaError_t e = launch_decode(p, d, dtype, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fwd_fp8_workspace_size(int B, int Hkv, int N, int d) {
  if (check_sizes(B, Hkv, Hkv, N, d, 1.0f, FA_BF16) != FA_OK || d != 128) return 0;
  const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  return (static_cast<size_t>(B) * Hkv * d * npad + 255) & ~size_t(255);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                     int d, int causal, float scale, float q_descale, float k_descale, float v_descale,
                     void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID;
  const fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, FA_BF16);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  for (float f : {q_descale, k_descale, v_descale})
    if (!(f > 0.f) || !std::isfinite(f)) return FA_ERR_INVALID;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < fa_fwd_fp8_workspace_size(B, Hkv, N, d))
    return FA_ERR_INVALID;
  Fp8Params p{};
  p.Npad = (N + 127) / 128 * 128;
  if (!encode_bshd_u8_map(&p.tm_q, q, B, N, Hq, d, 128) || !encode_bshd_u8_map(&p.tm_k, k, B, N, Hkv, d, 128) ||
      !encode_vt_u8_map(&p.tm_vt, workspace, B * Hkv, d, p.Npad))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  p.v = static_cast<const uint8_t*>(v);
  p.vt = static_cast<uint8_t*>(workspace);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.score_scale = scale * q_descale * k_descale;
  p.score_log2 = p.score_scale * 1.4426950408889634f;
  p.out_scale = v_descale;  // P and l both carry the 2^8 pre-scale, which cancels in O / l
  p.wait_limit_ns = kWaitLimitNs;
  const cudaError_t e = launch_fwd_fp8(p, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, const float* q_descale,
                                 const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq,
                                 int Hkv, int N, int d, int causal, float scale, void* workspace,
                                 size_t workspace_bytes, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID;
  if (q_descale == nullptr || k_descale == nullptr || v_descale == nullptr) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q_descale) | reinterpret_cast<uintptr_t>(k_descale) |
       reinterpret_cast<uintptr_t>(v_descale)) & 3u)
    return FA_ERR_INVALID;
  const fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, FA_BF16);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < fa_fwd_fp8_workspace_size(B, Hkv, N, d))
    return FA_ERR_INVALID;
  Fp8Params p{};
  p.Npad = (N + 127) / 128 * 128;
  if (!encode_bshd_u8_map(&p.tm_q, q, B, N, Hq, d, 128) || !encode_bshd_u8_map(&p.tm_k, k, B, N, Hkv, d, 128) ||
      !encode_vt_u8_map(&p.tm_vt, workspace, B * Hkv, d, p.Npad))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  p.v = static_cast<const uint8_t*>(v);
  p.vt = static_cast<uint8_t*>(workspace);
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.q_bs = q_descale;
  p.k_bs = k_descale;
  p.v_bs = v_descale;
  p.nb = (N + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  const cudaError_t e = launch_fwd_fp8(p, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                              const int* cache_seqlens, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                              int num_pages, int max_pages, int d, int causal, float scale, int num_splits,
                              fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID;
  if (!aligned4(cache_seqlens) || !aligned4(block_table)) return FA_ERR_INVALID;
  if (num_pages < 1 || max_pages < 1) return FA_ERR_INVALID;
  if (max_pages > (1 << 24) / 128) return FA_ERR_UNSUPPORTED;
  const int Nmax = max_pages * 128;
  const fa_status st = check_decode(B, Hq, Hkv, Nq, Nmax, d, scale, static_cast<int>(dtype), num_splits);
  if (st != FA_OK) return st;
  if (static_cast<long long>(num_pages) * 128 * Hkv * d * 2 >= (1LL << 40)) return FA_ERR_UNSUPPORTED;
  const DecodeSplit sp = decode_split(B, Hkv, Nmax, d, num_splits);
  const DecodeWorkspace ws = decode_workspace_layout(B, Hq, Hkv, Nq, Nmax, d, num_splits);
  if (ws.total > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                       workspace_bytes < ws.total))
    return FA_ERR_INVALID;
  const int G = Hq / Hkv;
  DecParams p{};
  if (!encode_bshd_box_map(&p.tm_q, q, B, Nq, Hq, d, G, Nq, dtype) ||
      !encode_bshd_map(&p.tm_k, k_pages, num_pages, 128, Hkv, d, 128, dtype) ||
      !encode_bshd_map(&p.tm_v, v_pages, num_pages, 128, Hkv, d, 128, dtype))
    return FA_ERR_CUDA;
  p.err = device_error_word();
  if (!p.err) return FA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  p.seqlens_k = cache_seqlens;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.opart = ws.total ? reinterpret_cast<float*>(w + ws.opart_off) : nullptr;
  p.lpart = ws.total ? reinterpret_cast<float*>(w + ws.lpart_off) : nullptr;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nmax = Nmax;
  p.G = G;
  p.M = G * Nq;
  p.S = sp.S;
  p.cps = sp.cps;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  const cudaError_t e = launch_decode(p, d, dtype, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_selftest_wait_timeout(int limit_us, fa_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_INVALID;
  unsigned* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  fa_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err,
                                                                               static_cast<uint64_t>(limit_us) * 1000);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_selftest_exp2(const float* x, float* y_poly, float* y_mufu, int n, fa_stream_t stream) {
  if (n < 0) return FA_ERR_INVALID;
  if (n == 0) return FA_OK;
  if (!aligned4(x) || !aligned4(y_poly) || !aligned4(y_mufu)) return FA_ERR_INVALID;
  const long long threads = (static_cast<long long>(n) + 1) / 2;
  const long long grid = (threads + 255) / 256;
  fa_selftest_exp2_kernel<<<static_cast<unsigned>(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      x, y_poly, y_mufu, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_check_device_error(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned* w = device_error_word();
  if (!w) return FA_ERR_CUDA;
  unsigned h = 0;
  if (cudaMemcpy(&h, w, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (h != 0) {
    const unsigned z = 0;
    if (cudaMemcpy(w, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    if (h & kDevErrTimeout) return FA_ERR_TIMEOUT;
    if (h & kDevErrSeqlens) return FA_ERR_INVALID;
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // extern "C"
