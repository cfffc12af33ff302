// noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd needs a caller-provided scratch workspace (per-row statistics and a float32
// dQ accumulator).  Some callers have no way to obtain one: a host framework whose
// caching allocator has already reserved the whole device, a plugin host that hands a
// kernel library only the tensors it operates on, or a latency-critical path where
// cudaMalloc -- which may synchronise the device and may fail -- is not acceptable.
// This entry point runs the same three backward launches as fa_bwd, with its scratch
// in a fixed array of device memory that belongs to the library.
//
// The array (kScratchBytes) is a file-scope __device__ variable, so every GPU on which
// the library's kernels are loaded holds it until the process exits.  Its device
// address is looked up on the first call made on that device, with that device
// current, and again whenever the current context of the device has changed since (a
// device reset replaces the context, and with it the array's address); that first
// call should therefore come before any stream capture.  All calls on a device share
// the one array and it keeps the last call's contents: the preprocess launch rewrites
// the statistics and zeroes the accumulator every call, and two calls whose work
// overlaps on the GPU (different streams, or different host threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "internal.h"

namespace fa {
namespace {

constexpr size_t kScratchBytes = 32ull << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // context each address was looked up in

// Device address of the scratch array on the current device, looked up on the first
// call in each context of the device.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

size_t fa_bwd_noalloc_max_scratch(void) { return fa::kScratchBytes; }

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dtype,
                   void* stream) {
  // Argument validation is fa_bwd's own: with no workspace it returns FA_ERR_WORKSPACE
  // only when every other argument is valid, and it launches nothing.
  const int st = fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, nullptr, 0, B, H, N, d, scale, causal, dtype, stream);
  if (st != FA_ERR_WORKSPACE) return st;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0 || need > fa::kScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int s2 = fa::scratch_for_current_device(&scratch);
  if (s2 != FA_OK) return s2;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, scratch, fa::kScratchBytes, B, H, N, d, scale, causal, dtype,
                stream);
}

}  // extern "C"
