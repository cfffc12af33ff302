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
  int pattern;                   // 0 dense, 1 butterfly block pattern (Nq = Nk, G = 1)
  float scale_log2;              // scale * log2(e)
  unsigned int* err_word;
  uint64_t limit_ns;
  int num_sms;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_do;       // {d, N, B*H}
  CUtensorMap tm_k, tm_v;        // {d, N, B*Hkv}
  CUtensorMap tm_dk, tm_dv;      // {d, N, B*Hkv}, box {64, 32, 1}, 128-byte swizzle: the dK/dV stores
  CUtensorMap tm_dq;  // 3-D map {d, N, B*H} over the float32 dQ accumulator, box {16, 32, 1}
                      // (64-byte swizzle), or {32, 32, 1} (128-byte swizzle) when wide_dq
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  uint8_t* stats;     // [B*H*Npad/128] 4 KB tiles: -lse/scale and -D per query row as three
                      // 16-bit terms each, the B operand of the rank-one MMAs (kStatsTileBytes)
  float* dq_accum;    // [B*H*N*d]   float32 dQ partial sums
  unsigned int* tile_counter;  // tiles handed out beyond the first one per CTA
  int BH, N, Npad, d, dtype, causal;   // BH = B*H query heads
  int BHkv, H, G;                      // B*Hkv key/value heads; G = H / Hkv query heads per key/value head
  int pattern;                         // 0 dense, 1 butterfly block pattern (G = 1)
  float scale, scale_log2;
  unsigned int* err_word;
  uint64_t limit_ns;
  int num_sms;
  int heads_per_group;           // tile order: see group_order
  int wide_dq;                   // d = 64, dense: dQ staged in 32-column chunks (one per warp)
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

// ---------------------------------------------------------------- butterfly block pattern
// Block-sparse attention with a fixed butterfly pattern on blocks of 256 rows / keys
// (pairs of 128-row tiles): pair p and pair q are linked iff p == q or p ^ q has exactly
// one bit set.  dir < 0 keeps only pairs <= p (causal forward: keys of a query pair),
// dir > 0 only pairs >= p (causal backward: queries of a key pair), dir == 0 all.
// Linked pairs in increasing order: p with one set bit cleared (highest bit first),
// p itself, p with one clear bit set (lowest bit first) while below npairs.
__host__ __device__ inline int bfly_count(int p, int npairs, int dir) {
  int n = 1;
  for (int b = 0; b < 31 && (1 << b) <= (p > npairs ? p : npairs); ++b) {
    const int c = p ^ (1 << b);
    if (c < p ? dir <= 0 : (dir >= 0 && c < npairs)) ++n;
  }
  return n;
}

__host__ __device__ inline int bfly_pair(int p, int i, int npairs, int dir) {
  if (dir <= 0) {
    for (int b = 30; b >= 0; --b)
      if ((p >> b) & 1) {
        if (i == 0) return p ^ (1 << b);
        --i;
      }
  }
  if (i == 0) return p;
  --i;
  for (int b = 0; b < 31 && (1 << b) < npairs; ++b)
    if (!((p >> b) & 1)) {
      const int c = p | (1 << b);
      if (c < npairs) {
        if (i == 0) return c;
        --i;
      }
    }
  return -1;
}

// The 128-row blocks of the linked pairs, in order: block j is half (j + skip) & 1 of
// linked pair (j + skip) >> 1.  skip = 1 drops the first block (the causal backward of an
// odd key block does not see the even query block of its own pair).  With an odd
// number of blocks the last pair holds one block; it is the largest pair, so when
// linked it is the last in the list and only the count changes.
__host__ __device__ inline int bfly_block(int p, int j, int npairs, int dir, int skip) {
  const int jj = j + skip;
  return 2 * bfly_pair(p, jj >> 1, npairs, dir) + (jj & 1);
}

__host__ __device__ inline int bfly_blocks(int p, int npairs, int nblocks, int dir, int skip) {
  const int cnt = bfly_count(p, npairs, dir);
  int n = 2 * cnt - skip;
  if ((nblocks & 1) && bfly_pair(p, cnt - 1, npairs, dir) == npairs - 1) --n;
  return n;
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

// Unique id of the calling thread's current CUDA context (0 when there is none or it
// cannot be read).  Device addresses of the library's __device__ variables are valid
// in the context they were looked up in; a device reset replaces the context.
unsigned long long current_context_id();

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
  CUtensorMap tm_k, tm_v;   // 3-D maps {d, Nk, B*Hkv}, box {64, 32, 1}, 128-byte swizzle
  unsigned int* err_word;   // bounded waits: error word and limit
  uint64_t limit_ns;
};
constexpr int kDecodeMaxRows = 8;
constexpr int kDecodeTmaKeys = 32;   // keys per stage of the split kernel
cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream);
// Backward stages: preprocess (D, lse2, zeroed accumulator), the dK/dV kernel with
// dQ partial sums, and the dQ conversion.
// Per 128-row query block the preprocess writes one tile of 128 rows x 16 16-bit values
// in the tensor core's K-major layout without swizzle (8-row x 16-byte core matrices, the
// two K halves 128 bytes apart, 8-row groups 256 bytes apart): K slots 0..2 hold
// -lse/scale split as 256*h + m + l, slots 8..10 hold -D split the same way, the rest 0.
constexpr int kStatsTileBytes = 4096;
constexpr int kBwdStagePre = 1;
constexpr int kBwdStageKV = 2;
constexpr int kBwdStageDQ = 4;
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stages);
cudaError_t launch_debug_wait(unsigned int* err_word, uint64_t limit_ns, cudaStream_t stream);

// FP8 (E4M3) forward, Nq = Nk, one key/value head per query head.
struct FwdF8Args {
  CUtensorMap tm_q, tm_k;   // 3-D maps {d, N, B*H} of 8-bit codes, box {d, 128, 1},
                            // 64-byte (d = 64) or 128-byte (d = 128) swizzle
  CUtensorMap tm_vt;        // 3-D map {N, d, B*H} over V^T (row stride Nt bytes), box {128, d, 1}
  const float* q_scale;     // [B*H, nb] per 128-row block
  const float* k_scale;
  const float* v_scale;
  void* o;                  // [B, H, N, d] 16-bit
  float* lse;
  int BH, N, d, dtype, causal;
  float scale_log2;
  unsigned int* err_word;
  uint64_t limit_ns;
  int num_sms;
};
cudaError_t launch_fwd_fp8(const FwdF8Args& a, cudaStream_t stream);

// E4M3 block quantization: per-block amax, scales, codes (three launches).
struct QuantArgs {
  const void* x;            // [B*H, N, d] 16-bit
  void* x8;                 // [B*H, N, d] codes, or [B*H, d, Nt] when transpose
  float* scales;            // [B*H, nb]
  const float* signs;       // [d] +-1, or nullptr for no rotation
  int BH, N, d, dtype, per_tensor, transpose, Nt;
};
cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream);

}  // namespace fa
