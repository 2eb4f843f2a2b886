// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs inside an engine or
// plugin that hands it only its input and output buffers, programs whose allocator is
// frozen after start-up (no cudaMalloc, no caching allocator), and real-time paths where a
// device allocation's latency or possible failure is not acceptable.  fa_bwd needs a
// caller-provided workspace; this entry point instead uses one scratch array that lives in
// the library itself, reserved when the library's device code is loaded on a GPU and held
// until the process exits.  It calls fa_bwd with that array, so the computation is
// exactly fa_bwd's.
#include "fa_internal.h"

#include <atomic>

namespace fa {
namespace {

constexpr size_t kNoallocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code its name is only a host-side stand-in: the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per device.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
  g_scratch_ptr[dev].store(addr, std::memory_order_release);
  return addr;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                    int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream) {
  const size_t need = fa_bwd_workspace_size(B, Hq, Hkv, N, d);
  if (need == 0) {
    // invalid or unsupported sizes: let fa_bwd report which, with a dummy workspace size
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype,
                  reinterpret_cast<void*>(uintptr_t(256)), 0, stream);
  }
  if (need > fa::kNoallocScratchBytes) return FA_ERR_UNSUPPORTED;
  void* scratch = fa::scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, scratch,
                fa::kNoallocScratchBytes, stream);
}
