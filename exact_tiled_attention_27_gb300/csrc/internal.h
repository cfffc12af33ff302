// internal.h -- declarations shared by the host API and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Device error word bits: bit 31 = a bounded wait gave up; the low bits name the site.
constexpr unsigned int kErrTimeoutBit = 0x80000000u;

// Default limit for one mbarrier wait inside a kernel (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct FwdArgs {
  CUtensorMap tm_q;              // 3-D map {d, Nq, B*H}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_k, tm_v;        // 3-D maps {d, Nk, B*Hkv}, same box and swizzle
  void* o;
  float* lse;
  int BH, H, G, Nq, Nk, d, dtype, causal;   // G = query heads per key/value head
  float scale_log2;              // scale * log2(e)
  unsigned int* err_word;
  uint64_t limit_ns;
  int num_sms;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_do;       // {d, N, B*H}
  CUtensorMap tm_k, tm_v;        // {d, N, B*Hkv}
  CUtensorMap tm_dq;  // 3-D map {d, N, B*H} over the float32 dQ accumulator, box {32, 128, 1}
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dvec;        // [B*H*Npad]  D = rowsum(dO o O), 0 on padding rows
  float* lse2;        // [B*H*Npad]  lse * log2(e), +inf on padding rows
  float* dq_accum;    // [B*H*N*d]   float32 dQ partial sums
  unsigned int* tile_counter;  // tiles handed out beyond the first one per CTA
  int BH, N, Npad, d, dtype, causal;   // BH = B*H query heads
  int BHkv, H, G;                      // B*Hkv key/value heads; G = H / Hkv query heads per key/value head
  float scale, scale_log2;
  unsigned int* err_word;
  uint64_t limit_ns;
  int num_sms;
  int heads_per_group;           // tile order: see group_order
};

// Order of the persistent work tiles.  A head (b, h) has `units` tiles, unit 0 the
// heaviest under the causal mask.  Heads are taken in groups of `hg`; inside a group
// the order is unit-major, so the CTAs running at any one time share the few heads
// of one group and the tensors those heads re-read stay in L2.  hg >= BH gives the
// plain unit-major order over all heads.
__host__ __device__ __forceinline__ void group_order(int tile, int BH, int units, int hg, int& r, int& bh) {
  const int per_group = hg * units;
  const int grp = tile / per_group;
  const int within = tile - grp * per_group;
  const int gh = (BH - grp * hg) < hg ? (BH - grp * hg) : hg;
  r = within / gh;
  bh = grp * hg + (within - r * gh);
}

// Heads per group so that `bytes_per_head` of re-read data for one group fits in
// half of the L2 cache (at least 1, at most BH).
inline int heads_per_group(long long bytes_per_head, long long l2_bytes, int BH) {
  long long g = (l2_bytes / 2) / (bytes_per_head > 0 ? bytes_per_head : 1);
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return static_cast<int>(g);
}

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel in the stream drains; every kernel here calls grid_dep_wait before
// it reads or writes global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);

// Split-key decode: the M = (H/Hkv)*Nq query rows of each key/value head (M <= 8)
// against Nk keys cut into S ranges of `chunk` keys; partial results in opart/lpart
// when S > 1.
struct DecArgs {
  const void* q;      // [B, H, Nq, d]
  const void* k;      // [B, Hkv, Nk, d]
  const void* v;
  void* o;            // [B, H, Nq, d]
  float* lse;         // [B, H, Nq]
  float* opart;       // [S, B*Hkv, M, d] float32 (S > 1)
  float* lpart;       // [S, B*Hkv, M] float32 natural-log lse of each range
  int BHkv, H, Hkv, Nq, Nk, M, S, chunk, d, dtype, causal;
  float scale_log2;
};
constexpr int kDecodeMaxRows = 8;
int decode_keys_per_step(int d);
cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream);
// Backward stages: preprocess (D, lse2, zeroed accumulator), the dK/dV kernel with
// dQ partial sums, and the dQ conversion.
constexpr int kBwdStagePre = 1;
constexpr int kBwdStageKV = 2;
constexpr int kBwdStageDQ = 4;
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stages);
cudaError_t launch_debug_wait(unsigned int* err_word, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fa
