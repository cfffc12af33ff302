// api.cu -- the C ABI declared in include/fa.h: argument validation, tensor-map
// encoding, workspace carving, launches and the device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// One error word per device: bit 31 set by a kernel whose bounded wait gave up.
__device__ unsigned int g_err_word;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  long long l2_bytes = 0;
  int major = 0;
  unsigned int* err_word = nullptr;
  unsigned long long ctx = 0;   // context the error word's address was looked up in
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Driver calls that identify the current context (resolved once through the runtime's
// entry-point query, so the library needs no link against the driver library).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void* driver_fn(const char* name, int version) {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return fn;
}

int get_device(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    if (prop.major != 10) return FA_ERR_NO_DEVICE;   // tcgen05 / TMEM need the sm_100 family
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.num_sms = prop.multiProcessorCount;
    d.l2_bytes = prop.l2CacheSize;
    d.major = prop.major;
    d.ready = true;
  }
  // The error word's device address belongs to the context it was looked up in; a
  // device reset (or a context the caller made current) gets a new one.
  const unsigned long long ctx = current_context_id();
  if (d.err_word == nullptr || ctx == 0 || ctx != d.ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    d.err_word = static_cast<unsigned int*>(p);
    d.ctx = current_context_id();   // the lookup creates the context if there was none
  }
  *out = &d;
  return FA_OK;
}

// 3-D map over a contiguous (B*H, N, d) 16-bit tensor: box of 128 rows x 64 elements
// (one 128-byte swizzle row per tensor row); rows past N read as zero.
bool encode_bhnd(CUtensorMap* m, const void* base, int BH, int N, int d, int dtype) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a contiguous (B*H, N, d) 16-bit tensor with a box of `rows` rows x 64
// elements, 128-byte swizzle (the decode kernel's 32-key stages).
bool encode_bhnd_rows(CUtensorMap* m, const void* base, int BH, int N, int d, int dtype, int rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, dtype == FA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the contiguous (B*H, N, d) float32 dQ accumulator: box of 32 rows x
// 16 floats (one 64-byte swizzle row per tensor row), used for bulk reductions.
bool encode_accum(CUtensorMap* m, void* base, int BH, int N, int d, bool wide) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  const cuuint32_t box[3] = {wide ? 32u : 16u, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over contiguous (B*H, N, d) E4M3 codes: box of 128 rows x d bytes, 64-byte
// swizzle at d = 64 and 128-byte at d = 128 (one swizzle row per tensor row).
bool encode_fp8_rows(CUtensorMap* m, const void* base, int BH, int N, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)N * d};
  const cuuint32_t box[3] = {(cuuint32_t)d, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over V^T codes (B*H, d, Nt): box of d rows x 128 keys, 128-byte swizzle; keys
// past N read as zero whatever the padding holds.
bool encode_fp8_vt(CUtensorMap* m, const void* base, int BH, int N, int Nt, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)d, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)Nt, (cuuint64_t)Nt * d};
  const cuuint32_t box[3] = {128, (cuuint32_t)d, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int fp8_vt_cols(int N) { return (N + 15) / 16 * 16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int N, int d, float scale, int dtype) {
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  const long long bhn = (long long)B * H * N;
  if ((long long)B * H > (1LL << 30) || bhn >= (1LL << 31) || bhn * d >= (1LL << 40)) return FA_ERR_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  return FA_OK;
}

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t sched_off, stats_off, acc_off, total;
  int Npad;
};

WsLayout ws_layout(int B, int H, int N, int d) {
  WsLayout w;
  w.Npad = (N + 127) / 128 * 128;
  const size_t blocks = (size_t)B * H * (w.Npad / 128);
  w.sched_off = 0;                        // tile counter of the dK/dV kernel
  w.stats_off = kAlign;                   // per-query-block statistics tiles
  w.acc_off = w.stats_off + round_up(blocks * kStatsTileBytes);
  w.total = w.acc_off + round_up((size_t)B * H * N * d * 4);
  return w;
}

// Test hook: wait on an mbarrier nobody arrives on, give up after the limit.
__global__ void debug_wait_kernel(unsigned int* err_word, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, err_word, limit_ns};
  mbar_wait(smem_u32(&bar), 0, ctl, 0x7ff);
  __syncthreads();
}

}  // namespace

unsigned long long current_context_id() {
  std::call_once(g_ctx_once, [] {
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent", 4000));
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId", 12000));
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current == nullptr || g_ctx_id == nullptr || g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr ||
      g_ctx_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

cudaError_t launch_debug_wait(unsigned int* err_word, uint64_t limit_ns, cudaStream_t stream) {
  debug_wait_kernel<<<1, 32, 0, stream>>>(err_word, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

extern "C" {

static int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                      int Nq, int Nk, int d, float scale, int causal, int dtype, void* stream, int pattern = 0) {
  int st = check_common(B, H, Nq, d, scale, dtype);
  if (st != FA_OK) return st;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_SHAPE;
  st = check_common(B, Hkv, Nk, d, scale, dtype);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  st = get_device(&dev);
  if (st != FA_OK) return st;
  FwdArgs a;
  const int BH = B * H;
  if (!encode_bhnd(&a.tm_q, q, BH, Nq, d, dtype) || !encode_bhnd(&a.tm_k, k, B * Hkv, Nk, d, dtype) ||
      !encode_bhnd(&a.tm_v, v, B * Hkv, Nk, d, dtype))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.H = H;
  a.G = H / Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.dtype = dtype;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err_word = dev->err_word;
  a.limit_ns = kWaitLimitNs;
  a.num_sms = dev->num_sms;
  a.pattern = pattern;
  return launch_fwd(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, float scale,
           int causal, int dtype, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, H, N, N, d, scale, causal, dtype, stream);
}

int fa_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
                 int Nk, int d, float scale, int causal, int dtype, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, dtype, stream);
}

int fa_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                  float scale, int causal, int pattern, int dtype, void* stream) {
  if (pattern != FA_PATTERN_BUTTERFLY) return FA_ERR_PATTERN;
  return fwd_common(q, k, v, o, lse, B, H, H, N, N, d, scale, causal, dtype, stream, 1);
}

int fa_fp8_vt_cols(int N) { return N >= 1 ? fp8_vt_cols(N) : 0; }

int fa_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, int dtype, const float* signs,
                    int per_tensor, int transpose, void* stream) {
  int st = check_common(B, H, N, d, 1.0f, dtype);
  if (st != FA_OK) return st;
  if (!x || !x8 || !scales) return FA_ERR_NULL;
  if (!aligned16(x) || !aligned16(x8) || (reinterpret_cast<uintptr_t>(scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(signs) & 3u))
    return FA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  st = get_device(&dev);
  if (st != FA_OK) return st;
  QuantArgs a;
  a.x = x;
  a.x8 = x8;
  a.scales = scales;
  a.signs = signs;
  a.BH = B * H;
  a.N = N;
  a.d = d;
  a.dtype = dtype;
  a.per_tensor = per_tensor ? 1 : 0;
  a.transpose = transpose ? 1 : 0;
  a.Nt = fp8_vt_cols(N);
  return launch_quantize_fp8(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
               int dtype, void* stream) {
  int st = check_common(B, H, N, d, scale, dtype);
  if (st != FA_OK) return st;
  if (!q8 || !k8 || !vt8 || !q_scale || !k_scale || !v_scale || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) ||
      ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
        reinterpret_cast<uintptr_t>(v_scale) | reinterpret_cast<uintptr_t>(lse)) & 3u))
    return FA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  st = get_device(&dev);
  if (st != FA_OK) return st;
  FwdF8Args a;
  const int BH = B * H;
  if (!encode_fp8_rows(&a.tm_q, q8, BH, N, d) || !encode_fp8_rows(&a.tm_k, k8, BH, N, d) ||
      !encode_fp8_vt(&a.tm_vt, vt8, BH, N, fp8_vt_cols(N), d))
    return FA_ERR_LAUNCH;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.d = d;
  a.dtype = dtype;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err_word = dev->err_word;
  a.limit_ns = kWaitLimitNs;
  a.num_sms = dev->num_sms;
  return launch_fwd_fp8(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_butterfly_blocks(int nblocks, int pair, int causal_dir, int* out, int cap) {
  const int npairs = (nblocks + 1) / 2;
  if (nblocks < 1 || pair < 0 || pair >= npairs || causal_dir < -1 || causal_dir > 1) return -1;
  const int n = bfly_blocks(pair, npairs, nblocks, causal_dir, 0);
  for (int j = 0; j < n && j < cap; ++j) out[j] = bfly_block(pair, j, npairs, causal_dir, 0);
  return n;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_common(B, H, N, d, 1.0f, FA_BF16) != FA_OK) return 0;
  return ws_layout(B, H, N, d).total;
}

static int bwd_common(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int Hkv, int N,
                      int d, float scale, int causal, int dtype, void* stream, int stages, int pattern = 0) {
  int st = check_common(B, H, N, d, scale, dtype);
  if (st != FA_OK) return st;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_SHAPE;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_ALIGN;
  const WsLayout w = ws_layout(B, H, N, d);
  if (workspace == nullptr || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return FA_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  st = get_device(&dev);
  if (st != FA_OK) return st;
  BwdArgs a;
  const int BH = B * H;
  if (!encode_bhnd(&a.tm_q, q, BH, N, d, dtype) || !encode_bhnd(&a.tm_k, k, B * Hkv, N, d, dtype) ||
      !encode_bhnd(&a.tm_v, v, B * Hkv, N, d, dtype) || !encode_bhnd(&a.tm_do, dO, BH, N, d, dtype) ||
      !encode_bhnd_rows(&a.tm_dk, dk, B * Hkv, N, d, dtype, 32) ||
      !encode_bhnd_rows(&a.tm_dv, dv, B * Hkv, N, d, dtype, 32))
    return FA_ERR_LAUNCH;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.tile_counter = reinterpret_cast<unsigned int*>(ws + w.sched_off);
  a.stats = ws + w.stats_off;
  a.dq_accum = reinterpret_cast<float*>(ws + w.acc_off);
  // d = 64, dense: long tiles stage dQ in 32-column chunks (half as many bulk reductions,
  // one staging chunk per warp); short tiles keep 16-column chunks, two per warp in flight
  const int nb = (N + 127) / 128;
  const int steps_per_tile = causal ? (nb + 1) / 2 : nb;
  a.wide_dq = (d == 64 && pattern == 0 && Hkv == H && steps_per_tile >= 24) ? 1 : 0;
  if (!encode_accum(&a.tm_dq, a.dq_accum, BH, N, d, a.wide_dq != 0)) return FA_ERR_LAUNCH;
  a.BH = BH;
  a.BHkv = B * Hkv;
  a.H = H;
  a.G = H / Hkv;
  a.N = N;
  a.Npad = w.Npad;
  a.d = d;
  a.dtype = dtype;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err_word = dev->err_word;
  a.limit_ns = kWaitLimitNs;
  a.num_sms = dev->num_sms;
  // every key block re-reads the Q and dO (16-bit) of the key/value head's G query heads
  // and adds into their float32 dQ
  a.heads_per_group = heads_per_group(8LL * a.G * N * d, dev->l2_bytes, a.BHkv);
  a.pattern = pattern;
  return launch_bwd(a, static_cast<cudaStream_t>(stream), stages) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
           void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d, float scale, int causal,
           int dtype, void* stream) {
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale, causal, dtype, stream,
                    kBwdStagePre | kBwdStageKV | kBwdStageDQ);
}

int fa_bwd_preprocess(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                      float scale, int causal, int dtype, void* stream) {
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale, causal, dtype, stream,
                    kBwdStagePre);
}

int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                float scale, int causal, int dtype, void* stream) {
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale, causal, dtype, stream,
                    kBwdStageKV);
}

int fa_bwd_dq_convert(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                      float scale, int causal, int dtype, void* stream) {
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale, causal, dtype, stream,
                    kBwdStageDQ);
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int Hkv, int N, int d,
               float scale, int causal, int dtype, void* stream) {
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, Hkv, N, d, scale, causal, dtype,
                    stream, kBwdStagePre | kBwdStageKV | kBwdStageDQ);
}

// ---------------------------------------------------------------- split-key decode
// Ranges hold at least 256 keys; at most 128 ranges.
static int decode_max_splits(int Nk) {
  int s = Nk / 256;
  return s < 1 ? 1 : (s > 128 ? 128 : s);
}

static int decode_check(int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int dtype) {
  int st = check_common(B, H, Nq, d, scale, dtype);
  if (st != FA_OK) return st;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_SHAPE;
  st = check_common(B, Hkv, Nk, d, scale, dtype);
  if (st != FA_OK) return st;
  if ((long long)(H / Hkv) * Nq > kDecodeMaxRows) return FA_ERR_SHAPE;
  if ((long long)B * Hkv > 65535) return FA_ERR_SHAPE;   // one grid row per key/value head
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
  if (decode_check(B, H, Hkv, Nq, Nk, d, 1.0f, FA_BF16) != FA_OK) return 0;
  const int smax = decode_max_splits(Nk);
  if (smax == 1) return 0;
  const size_t rows = (size_t)smax * B * Hkv * (H / Hkv) * Nq;
  return round_up(rows * d * 4) + round_up(rows * 4);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, size_t ws_bytes,
              int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal, int dtype, void* stream) {
  int st = decode_check(B, H, Hkv, Nq, Nk, d, scale, dtype);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_ALIGN;
  const size_t need = fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d);
  if (need > 0 && (workspace == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))))
    return FA_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  st = get_device(&dev);
  if (st != FA_OK) return st;
  DecArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.BHkv = B * Hkv;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.M = (H / Hkv) * Nq;
  a.d = d;
  a.dtype = dtype;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err_word = dev->err_word;
  a.limit_ns = kWaitLimitNs;
  if (!encode_bhnd_rows(&a.tm_k, k, a.BHkv, Nk, d, dtype, kDecodeTmaKeys) ||
      !encode_bhnd_rows(&a.tm_v, v, a.BHkv, Nk, d, dtype, kDecodeTmaKeys))
    return FA_ERR_LAUNCH;
  // One CTA per SM at a time.  The number of ranges minimises the makespan estimate
  // (waves of CTAs x stages per range, plus a few stages of start-up), with ranges of at
  // least 8 stages.
  const int smax = decode_max_splits(Nk);
  const long long stages = (Nk + kDecodeTmaKeys - 1) / kDecodeTmaKeys;
  long long best = -1;
  int best_s = 1;
  for (int sp = 1; sp <= smax; ++sp) {
    const long long per = (stages + sp - 1) / sp;
    if (sp > 1 && per < 8) break;
    const long long waves = ((long long)a.BHkv * sp + dev->num_sms - 1) / dev->num_sms;
    const long long cost = waves * (per + 4);
    if (best < 0 || cost < best) {
      best = cost;
      best_s = sp;
    }
  }
  const long long per = (stages + best_s - 1) / best_s;
  a.chunk = (int)(per * kDecodeTmaKeys);
  a.S = (Nk + a.chunk - 1) / a.chunk;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = (size_t)a.S * a.BHkv * a.M;
  a.opart = a.S > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  a.lpart = a.S > 1 ? reinterpret_cast<float*>(ws + round_up(rows * d * 4)) : nullptr;
  return launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd_sparse(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                  float scale, int causal, int pattern, int dtype, void* stream) {
  if (pattern != FA_PATTERN_BUTTERFLY) return FA_ERR_PATTERN;
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale, causal, dtype,
                    stream, kBwdStagePre | kBwdStageKV | kBwdStageDQ, 1);
}

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "B, H and N must be >= 1, B*H <= 2^30 and B*H*N < 2^31";
    case FA_ERR_UNSUPPORTED_D: return "head_dim must be 64 or 128";
    case FA_ERR_DTYPE: return "dtype must be FA_BF16 or FA_FP16";
    case FA_ERR_ALIGN: return "tensor base addresses must be 16-byte aligned (lse: 4-byte)";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned (256 bytes) or smaller than fa_bwd_workspace_size";
    case FA_ERR_LAUNCH: return "the CUDA runtime rejected a launch";
    case FA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded pipeline wait gave up";
    case FA_ERR_NO_DEVICE: return "no usable sm_100-family CUDA device is current";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_PATTERN: return "unknown block pattern (FA_PATTERN_BUTTERFLY is the only one)";
    case FA_ERR_SCRATCH_LIMIT:
      return "fa_bwd_noalloc: these sizes need more scratch than its built-in array (fa_bwd_noalloc_max_scratch)";
    default: return "unknown status";
  }
}

int fa_get_last_kernel_status(void* stream) {
  DeviceInfo* dev = nullptr;
  int st = get_device(&dev);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return (word & kErrTimeoutBit) ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

int fa_device_sm_count(void) {
  DeviceInfo* dev = nullptr;
  const int st = get_device(&dev);
  return st == FA_OK ? dev->num_sms : -st;
}

int fa_debug_wait_timeout(unsigned limit_us, void* stream) {
  DeviceInfo* dev = nullptr;
  const int st = get_device(&dev);
  if (st != FA_OK) return st;
  if (limit_us < 1) limit_us = 1;
  if (limit_us > 2000000) limit_us = 2000000;
  return launch_debug_wait(dev->err_word, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

}  // extern "C"
