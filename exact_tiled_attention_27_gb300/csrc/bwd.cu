// bwd.cu -- backward kernels of exact tiled attention for sm_103a.
//
// The backward recomputes the probabilities on chip from Q, K and the saved row
// log-sum-exp instead of reading a stored N x N matrix (review of the FlashAttention
// paper, "方法细节"; "Flash Attention" chapter, end of "FlashAttention——把整件事分块
// 塞进 SRAM").  Gradient formulas are the derivative of O = softmax(scale Q K^T) V:
//
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Three launches:
//   bwd_pre_kernel   -lse/scale and -D per query row, each split into three 16-bit
//                    terms and written as one operand tile per 128-row block (zeros
//                    on padding rows, whose Q and dO rows read as zero); zeroes the
//                    float32 dQ accumulator.
//   bwd_kv_kernel    persistent over (batch*head, 128-key block) tiles, key/value
//                    block on the outside, query blocks inside.  Per query block:
//                      S^T - lse/scale = K Q^T + 1 (-lse/scale)^T,
//                      dP^T - D = V dO^T + 1 (-D)^T          (tcgen05, tensor memory;
//                                        the per-query statistics enter as one more
//                                        rank-one MMA each, so no thread loads them)
//                      P^T = 2^((S^T - lse/scale) scale log2e), dS^T = P^T o (dP^T - D)
//                                        (one thread per key row and query half)
//                      dV += P^T dO      (P^T read from tensor memory)
//                      dK += dS^T Q, dQ_part = dS K      (dS^T from shared memory)
//                    dQ_part is added into the float32 accumulator by bulk tensor
//                    reductions; dK (times scale) and dV are written once per tile.
//   bwd_dq_kernel    dq = scale * accumulator, rounded to the 16-bit type.
//
// Warp roles of bwd_kv_kernel (16 warps, registers re-split with setmaxnreg):
//   warps 0-3, 4-7   dS warpgroups: key row = lane of tensor memory; warpgroup h
//                    handles query columns 64h .. 64h+63 of the current block
//   warps 8-11       dQ warpgroup: copies dQ_part from tensor memory into a swizzled
//                    shared-memory tile that one thread adds into the float32
//                    accumulator with a bulk tensor reduction (whole 128-byte
//                    lines, done by the copy engine); writes dK and dV at the end
//                    of a tile (on short d = 64 tiles staged in the same ring and
//                    written by bulk tensor stores)
//   warp 12          TMA producer; warp 13 MMA issuer; warps 14-15 idle
//
// At d = 64 the tensor-memory columns hold S^T, dP^T, dV, dK, dQ and P^T side by side,
// and the next block's S^T / dP^T are issued as soon as the dS warpgroups have read
// the current ones, so the tensor core computes them while dS is formed.  At d = 128
// (512 columns are taken by S^T, dP^T, dV, dK) P^T shares the S^T columns and dQ
// shares the dP^T columns, and the steps run in order.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRows = 128;
constexpr int kChunkBytes = kRows * 128;
constexpr int kBwdThreads = 512;
constexpr int kBwdLaunchRegs = 128;
// Register split (setmaxnreg) per warpgroup: the two dS warpgroups, the dQ warpgroup and
// the control warps (producer, MMA issuer).  At d = 128 the dQ warpgroup gets 112 (its
// 64 columns of dQ per staging round and the dK/dV read-out spilled at 96) and the control
// warps 80: +7.6 % on the d = 128 backward.  At d = 64 the same split measured 2 % slower,
// so it keeps 96 / 96.
constexpr int kDsRegs = 160;
template <int D>
constexpr int kDqRegs = D == 128 ? 112 : 96;
template <int D>
constexpr int kCtlRegs = D == 128 ? 80 : 96;
static_assert((2 * kDsRegs + kDqRegs<64> + kCtlRegs<64>) * 128 <= kBwdLaunchRegs * kBwdThreads &&
                  (2 * kDsRegs + kDqRegs<128> + kCtlRegs<128>) * 128 <= kBwdLaunchRegs * kBwdThreads,
              "register split exceeds the launch");
constexpr int kTileSlots = 4;   // tile numbers the producer may publish ahead of the slowest role

template <int D, bool WIDE = false>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kRows * D * 2;
  static constexpr bool kEarly = (D == 64);          // next S^T / dP^T issued before this block's gradients
  static constexpr int kKVBufs = (D == 64) ? 2 : 1;
  static constexpr int kQBufs = (D == 64) ? 3 : 1;
  // dQ staging: every warp of the dQ warpgroup stages its 32 rows in chunks of 16 floats
  // (2 KB, 64-byte swizzle) through a ring of its own, so that a chunk is written while
  // the bulk reductions of the previous ones still read theirs (16 KB at d = 64, which
  // leaves room for the third Q/dO buffer; 32 KB at d = 128)
  // (WIDE, d = 64 only: 32 rows x 32 floats, 4 KB, 128-byte swizzle, one per warp: half as
  // many bulk reductions, which measured faster on long tiles and slower on short ones)
  static_assert(!WIDE || D == 64, "wide dQ staging is a d = 64 layout");
  static constexpr int kDQCols = WIDE ? 32 : 16;
  static constexpr int kDQRing = WIDE ? 1 : ((D == 64) ? 2 : 4);
  static constexpr int kDQChunkBytes = 32 * kDQCols * 4;
  static_assert(!kEarly || kQBufs >= 2, "early issue needs two Q/dO buffers");
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVBufs * kTileBytes;
  static constexpr int kOffQ = kOffV + kKVBufs * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQBufs * kTileBytes;
  static constexpr int kOffDST = kOffDO + kQBufs * kTileBytes;       // 128 x 128 16-bit, K-major SW128
  static constexpr int kOffDQS = kOffDST + 2 * kChunkBytes;          // dQ staging: [4 warps][kDQRing] chunks
  static constexpr int kOffStats = kOffDQS + 4 * kDQRing * kDQChunkBytes;   // [kQBufs] statistics tiles
  // constant A operands of the rank-one MMAs, three 8-row x 16-byte core matrices
  // [C | 0 | C], C = (256, 1, 1, 0, 0, 0, 0, 0) in every row: A_L = (C, 0) picks K slots
  // 0..2 of a statistics tile (-lse/scale), A_D = (0, C) slots 8..10 (-D)
  static constexpr int kOffCoef = kOffStats + kQBufs * kStatsTileBytes;
  static constexpr int kOffRing = kOffCoef + 3 * 128;   // int[kTileSlots]
  static constexpr int kOffBar = kOffRing + kTileSlots * 4;
  // barriers
  static constexpr int kKVFull = 0;                   // [kKVBufs]
  static constexpr int kKVEmpty = kKVFull + kKVBufs;  // [kKVBufs]
  static constexpr int kQFull = kKVEmpty + kKVBufs;   // [kQBufs]
  static constexpr int kQEmpty = kQFull + kQBufs;     // [kQBufs]
  static constexpr int kSFull = kQEmpty + kQBufs;
  static constexpr int kSTFree = kSFull + 1;
  static constexpr int kDSFull = kSTFree + 1;
  static constexpr int kMmaDone = kDSFull + 1;
  static constexpr int kDQFull = kMmaDone + 1;
  static constexpr int kDQFree = kDQFull + 1;
  static constexpr int kDKVFull = kDQFree + 1;
  static constexpr int kDKVEmpty = kDKVFull + 1;
  static constexpr int kTileFull = kDKVEmpty + 1;     // [kTileSlots]
  static constexpr int kTileEmpty = kTileFull + kTileSlots;   // [kTileSlots]
  static constexpr int kDrain = kTileEmpty + kTileSlots;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  // tensor memory columns (512 allocated)
  static constexpr uint32_t kTmST = 0;
  static constexpr uint32_t kTmDPT = 128;
  static constexpr uint32_t kTmDV = 256;
  static constexpr uint32_t kTmDK = 256 + D;
  static constexpr uint32_t kTmDQ = (D == 64) ? 384 : 128;
  // P^T (16-bit pairs along the query dimension), query half h
  __host__ __device__ static constexpr uint32_t tm_pt(int h) { return D == 64 ? 448 + 32 * h : 64 * h; }
};

// 16-byte unit `u` (8 elements) of row `r` inside a 128-row x 128-byte swizzled block.
__device__ __forceinline__ uint32_t sw128_offset(int r, int u) {
  return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

// MODE 1 (GQA): key/value heads shared by groups of G > 1 query heads (fa_bwd_gqa).
// MODE 2 (SPARSE): the butterfly block pattern (fa_bwd_sparse): a key block visits the
// query blocks of its pair's linked pairs.  MODE 0: G = 1, dense.  WIDE: 32-column dQ
// staging chunks (d = 64).
template <int D, int DT, bool CAUSAL, int MODE, bool WIDE>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, const uint8_t* __restrict__ stats, float* __restrict__ dq_accum,
                  unsigned int* __restrict__ tile_counter,
                  uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, int BHkv, int H, int G, int N, int Npad,
                  float scale,
                  float scale_log2, int hg, unsigned int* err_word, uint64_t limit_ns) {
  using C = BwdCfg<D, WIDE>;
  // dK/dV written through the dQ staging ring by bulk tensor stores on short tiles at d = 64
  // (the tile-end read-out is then off the dQ warpgroup's load/store pipe)
  constexpr bool kStagedDKV = D == 64 && !WIDE;
  // short d = 64 tiles: the next tile is claimed a tile ahead and its first scores are
  // issued during the current tile's last step when its operands are already in place
  constexpr bool kAhead = C::kKVBufs == 2 && !WIDE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so
  // that every access through it stays a shared-memory access (not a generic one)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  // warp index through a shuffle so the compiler can treat it as warp-uniform
  const int warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const int nb = (N + kRows - 1) / kRows;
  const int ntiles = BHkv * nb;   // (batch x key/value head, key block)
  // The query heads that read key/value head bhk are G consecutive heads starting at
  // first_q_head(bhk); a tile's steps run over all of their query blocks, so dK and dV
  // sum over the group in tensor memory.  G = 1 is ordinary multi-head attention.
  constexpr bool GQA = MODE == 1;
  constexpr bool SPARSE = MODE == 2;
  auto first_q_head = [&](int bhk) { return GQA ? (bhk / (H / G)) * H + (bhk % (H / G)) * G : bhk; };
  const int group = GQA ? G : 1;
  // butterfly lists of a key block: its pair, upward under the causal mask, without the
  // even query block of its own pair when the key block is odd (that block lies above
  // the diagonal)
  const int npairs = (nb + 1) >> 1;
  constexpr int kDir = CAUSAL ? 1 : 0;
  auto skip_of = [&](int kb) { return (CAUSAL && (kb & 1)) ? 1 : 0; };
  auto sparse_q = [&](int kb, int j) { return bfly_block(kb >> 1, j, npairs, kDir, skip_of(kb)); };
  auto sparse_n = [&](int kb) { return bfly_blocks(kb >> 1, npairs, nb, kDir, skip_of(kb)); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kKVBufs; ++i) {
      mbar_init(bar(C::kKVFull + i), 1);
      mbar_init(bar(C::kKVEmpty + i), 1);
    }
    for (int i = 0; i < C::kQBufs; ++i) {
      mbar_init(bar(C::kQFull + i), 1);
      mbar_init(bar(C::kQEmpty + i), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSTFree), 2 * kRows);
    mbar_init(bar(C::kDSFull), 2 * kRows);
    mbar_init(bar(C::kMmaDone), 1);
    mbar_init(bar(C::kDQFull), 1);
    mbar_init(bar(C::kDQFree), kRows);
    mbar_init(bar(C::kDKVFull), 1);
    mbar_init(bar(C::kDKVEmpty), kRows);
    for (int i = 0; i < kTileSlots; ++i) {
      mbar_init(bar(C::kTileFull + i), 1);
      mbar_init(bar(C::kTileEmpty + i), 13);   // every warp but the producer and the two idle ones
    }
    mbar_init(bar(C::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 3 * 8) {
    // the coefficient rows of the rank-one MMAs (16-bit 256 and 1)
    const uint32_t hi = (DT == 1) ? 0x5C00u : 0x4380u, one = (DT == 1) ? 0x3C00u : 0x3F80u;
    const bool c = (threadIdx.x >> 3) != 1;
    *reinterpret_cast<uint4*>(smem + C::kOffCoef + threadIdx.x * 16) =
        c ? make_uint4(hi | (one << 16), one, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl ctl{abort_flag, err_word, limit_ns};
  const WaitCtl drain{nullptr, err_word, limit_ns};
  // the set-up above overlapped the previous kernel's tail; global memory only from here.
  // (This grid does not release its dependents early: a dependent grid launched while
  // these CTAs run measurably slowed them down.)
  grid_dep_wait();

  // Work tiles: CTA c starts with tile c; the producer warp claims each further tile
  // from the global counter (heaviest tiles come first in tile order, so this is list
  // scheduling by decreasing cost) and publishes it to the other roles through a small
  // ring in shared memory.  -1 ends the loop.
  int* tile_ring = reinterpret_cast<int*>(smem + C::kOffRing);
  auto take_tile = [&](int k, uint32_t site) -> int {
    const int slot = k % kTileSlots;
    if (!wait_warp(bar(C::kTileFull + slot), (k / kTileSlots) & 1, ctl, site)) return -1;
    const int tile = reinterpret_cast<volatile int*>(tile_ring)[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar(C::kTileEmpty + slot));
    return tile;
  };

  if (warp >= 12) {
    regs_dec<kCtlRegs<D>>();
    if (warp == 12) {
      // ---------------------------------------------------------- TMA producer (whole warp; one lane issues)
      if (elect_one()) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
      }
      uint32_t s = 0;
      int it = 0;
      bool ok = true;
      if constexpr (kAhead) {
        // short d = 64 tiles: the tile after the current one is claimed as soon as the current
        // one starts, and its K and V go into the other buffer as soon as that buffer is free
        // (checked between this tile's Q/dO loads, waited for at its end), so that the MMA warp
        // can issue the next tile's first scores during this tile's last step
        auto publish = [&](int k, int tile) -> bool {
          const int slot = k % kTileSlots;
          if (k >= kTileSlots && !wait_warp(bar(C::kTileEmpty + slot), ((k / kTileSlots) - 1) & 1, ctl, 0x403))
            return false;
          if ((threadIdx.x & 31) == 0) {
            tile_ring[slot] = tile;
            mbar_arrive(bar(C::kTileFull + slot));   // release: the ring entry is visible with the phase
          }
          __syncwarp();
          return true;
        };
        auto issue_kv = [&](int k, int tile) {      // K and V of tile number k into buffer k % 2
          int kb, bh;
          group_order(tile, BHkv, nb, hg, kb, bh);
          const int kvb = k % C::kKVBufs;
          const uint32_t kdst = smem_u32(smem + C::kOffK + kvb * C::kTileBytes);
          const uint32_t vdst = smem_u32(smem + C::kOffV + kvb * C::kTileBytes);
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(C::kKVFull + kvb), 2 * C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              tma_load_3d(kdst + c * kChunkBytes, &tm_k, bar(C::kKVFull + kvb), c * 64, kb * kRows, bh);
              tma_load_3d(vdst + c * kChunkBytes, &tm_v, bar(C::kKVFull + kvb), c * 64, kb * kRows, bh);
            }
          }
          __syncwarp();
        };
        // buffer of tile number k free (the tile two earlier done with it); without blocking
        // unless `block`: 1 free, 0 not yet, -1 the wait gave up
        auto kv_free = [&](int k, bool block) -> int {
          if (k < C::kKVBufs) return 1;
          const uint32_t eb = bar(C::kKVEmpty + k % C::kKVBufs), par = ((k / C::kKVBufs) - 1) & 1;
          if (block) return wait_warp(eb, par, ctl, 0x401) ? 1 : -1;
          return __all_sync(0xffffffffu, mbar_test(eb, par) != 0u) ? 1 : 0;
        };
        int kv_done = 0;   // tile numbers whose K and V were issued
        int cur = static_cast<int>(blockIdx.x) < ntiles ? static_cast<int>(blockIdx.x) : -1;
        ok = publish(0, cur);
        if (ok && cur >= 0) {
          issue_kv(0, cur);
          kv_done = 1;
        }
        for (; ok && cur >= 0; ++it) {
          unsigned int claim = 0;
          if ((threadIdx.x & 31) == 0) claim = atomicAdd(tile_counter, 1u);
          int nxt = static_cast<int>(gridDim.x + __shfl_sync(0xffffffffu, claim, 0));
          if (nxt >= ntiles) nxt = -1;
          if (!publish(it + 1, nxt)) {
            ok = false;
            break;
          }
          int kb, bh;
          group_order(cur, BHkv, nb, hg, kb, bh);
          const int q0 = SPARSE ? sparse_q(kb, 0) : (CAUSAL ? kb : 0);
          const int nq = SPARSE ? sparse_n(kb) : 0;
          for (int g = 0; ok && g < group; ++g) {
          const int bhq = first_q_head(bh) + g;
          for (int qi = q0, j = 0; SPARSE ? j < nq : qi < nb; ++s, ++j, qi = SPARSE ? sparse_q(kb, j) : qi + 1) {
            if (nxt >= 0 && kv_done == it + 1 && kv_free(it + 1, false) == 1) {
              issue_kv(it + 1, nxt);
              kv_done = it + 2;
            }
            const int qs = s % C::kQBufs;
            if (s >= (uint32_t)C::kQBufs && !wait_warp(bar(C::kQEmpty + qs), ((s / C::kQBufs) - 1) & 1, ctl, 0x402)) {
              ok = false;
              break;
            }
            const uint32_t qdst = smem_u32(smem + C::kOffQ + qs * C::kTileBytes);
            const uint32_t odst = smem_u32(smem + C::kOffDO + qs * C::kTileBytes);
            const uint32_t sdst = smem_u32(smem + C::kOffStats + qs * kStatsTileBytes);
            if (elect_one()) {
              mbar_arrive_expect_tx(bar(C::kQFull + qs), 2 * C::kTileBytes + kStatsTileBytes);
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(qdst + c * kChunkBytes, &tm_q, bar(C::kQFull + qs), c * 64, qi * kRows, bhq);
                tma_load_3d(odst + c * kChunkBytes, &tm_do, bar(C::kQFull + qs), c * 64, qi * kRows, bhq);
              }
              const size_t sblock = (size_t)bhq * (Npad / kRows) + qi;
              bulk_load(sdst, stats + sblock * kStatsTileBytes, kStatsTileBytes, bar(C::kQFull + qs));
            }
            __syncwarp();
          }
          }
          if (!ok) break;
          if (nxt >= 0 && kv_done == it + 1) {
            if (kv_free(it + 1, true) != 1) {
              ok = false;
              break;
            }
            issue_kv(it + 1, nxt);
            kv_done = it + 2;
          }
          cur = nxt;
        }
        it = kv_done;   // the drain below waits for every K/V load issued
      } else {
      int next = static_cast<int>(blockIdx.x);
      for (;; ++it) {
        const int slot = it % kTileSlots;
        if (it >= kTileSlots && !wait_warp(bar(C::kTileEmpty + slot), ((it / kTileSlots) - 1) & 1, ctl, 0x403)) {
          ok = false;
          break;
        }
        const int tile = next < ntiles ? next : -1;
        if ((threadIdx.x & 31) == 0) {
          tile_ring[slot] = tile;
          mbar_arrive(bar(C::kTileFull + slot));   // release: the ring entry is visible with the phase
        }
        __syncwarp();
        if (tile < 0) break;
        int kb, bh;                        // key block: kb = 0 carries the most query blocks (causal)
        group_order(tile, BHkv, nb, hg, kb, bh);
        const int kvb = it % C::kKVBufs;
        if (it >= C::kKVBufs && !wait_warp(bar(C::kKVEmpty + kvb), ((it / C::kKVBufs) - 1) & 1, ctl, 0x401)) {
          ok = false;
          break;
        }
        const uint32_t kdst = smem_u32(smem + C::kOffK + kvb * C::kTileBytes);
        const uint32_t vdst = smem_u32(smem + C::kOffV + kvb * C::kTileBytes);
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::kKVFull + kvb), 2 * C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_3d(kdst + c * kChunkBytes, &tm_k, bar(C::kKVFull + kvb), c * 64, kb * kRows, bh);
            tma_load_3d(vdst + c * kChunkBytes, &tm_v, bar(C::kKVFull + kvb), c * 64, kb * kRows, bh);
          }
        }
        __syncwarp();
        const int q0 = SPARSE ? sparse_q(kb, 0) : (CAUSAL ? kb : 0);
        const int nq = SPARSE ? sparse_n(kb) : 0;
        for (int g = 0; ok && g < group; ++g) {
        const int bhq = first_q_head(bh) + g;
        for (int qi = q0, j = 0; SPARSE ? j < nq : qi < nb; ++s, ++j, qi = SPARSE ? sparse_q(kb, j) : qi + 1) {
          const int qs = s % C::kQBufs;
          if (s >= (uint32_t)C::kQBufs && !wait_warp(bar(C::kQEmpty + qs), ((s / C::kQBufs) - 1) & 1, ctl, 0x402)) {
            ok = false;
            break;
          }
          const uint32_t qdst = smem_u32(smem + C::kOffQ + qs * C::kTileBytes);
          const uint32_t odst = smem_u32(smem + C::kOffDO + qs * C::kTileBytes);
          const uint32_t sdst = smem_u32(smem + C::kOffStats + qs * kStatsTileBytes);
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(C::kQFull + qs), 2 * C::kTileBytes + kStatsTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              tma_load_3d(qdst + c * kChunkBytes, &tm_q, bar(C::kQFull + qs), c * 64, qi * kRows, bhq);
              tma_load_3d(odst + c * kChunkBytes, &tm_do, bar(C::kQFull + qs), c * 64, qi * kRows, bhq);
            }
            const size_t sblock = (size_t)bhq * (Npad / kRows) + qi;
            bulk_load(sdst, stats + sblock * kStatsTileBytes, kStatsTileBytes, bar(C::kQFull + qs));
          }
          __syncwarp();
        }
        }
        if (!ok) {
          ++it;   // this tile's K and V were issued: the drain below must wait for them
          break;
        }
        // claim the next tile only now, when this tile's last loads are issued and its
        // compute is about to end: the order of claims then follows the order in which
        // CTAs run out of work (list scheduling), not the order in which they started
        unsigned int claim = 0;
        if ((threadIdx.x & 31) == 0) claim = atomicAdd(tile_counter, 1u);
        next = static_cast<int>(gridDim.x + __shfl_sync(0xffffffffu, claim, 0));
      }
      }
      if (!ok) {
        // let every copy already issued land before the CTA exits
        for (int b = 0; b < C::kKVBufs; ++b)
          if (it > b) {
            const int last = it - 1 - ((it - 1 - b) % C::kKVBufs);
            mbar_wait(bar(C::kKVFull + b), (last / C::kKVBufs) & 1, drain, 0x4f1);
          }
        for (int b = 0; b < C::kQBufs; ++b)
          if (s > (uint32_t)b) {
            const uint32_t last = s - 1 - ((s - 1 - b) % C::kQBufs);
            mbar_wait(bar(C::kQFull + b), (last / C::kQBufs) & 1, drain, 0x4f2);
          }
      }
    } else if (warp == 13) {
      // ---------------------------------------------------------- MMA issuer (whole warp; one lane issues)
      constexpr uint32_t ab = (DT == 0) ? 1u : 0u;
      constexpr uint32_t idesc_s = idesc_f16(ab, 0, 0, 128, 128);    // A, B K-major
      constexpr uint32_t idesc_kv = idesc_f16(ab, 0, 1, 128, D);     // A K-major, B MN-major
      constexpr uint32_t idesc_q = idesc_f16(ab, 1, 1, 128, D);      // A MN-major, B MN-major
      const uint32_t dst = smem_u32(smem + C::kOffDST);
      auto qaddr = [&](uint32_t step) { return smem_u32(smem + C::kOffQ + (step % C::kQBufs) * C::kTileBytes); };
      auto oaddr = [&](uint32_t step) { return smem_u32(smem + C::kOffDO + (step % C::kQBufs) * C::kTileBytes); };
      // S^T = K Q^T and / or dP^T = V dO^T (A, B K-major, 16 elements = 32 bytes per step)
      auto issue_st = [&](uint32_t kbase, uint32_t qbase) {
        const uint64_t kd = sdesc_sw128(kbase, 16, 1024), qd = sdesc_sw128(qbase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          umma_ss(tmem + C::kTmST, kd + off, qd + off, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dpt = [&](uint32_t vbase, uint32_t obase) {
        const uint64_t vd = sdesc_sw128(vbase, 16, 1024), od = sdesc_sw128(obase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          umma_ss(tmem + C::kTmDPT, vd + off, od + off, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      // the per-query statistics of step `step` added to every key row: S^T += 1 (-lse/scale)^T
      // and dP^T += 1 (-D)^T, A = a constant coefficient block (all 8-row groups read the same
      // core matrix: stride 0), B = the statistics tile (K-major, no swizzle)
      const uint32_t coef = smem_u32(smem + C::kOffCoef);
      const uint64_t a_lse = sdesc_noswz(coef, 128, 0);
      const uint64_t a_d = sdesc_noswz(coef + 128, 128, 0);
      auto stats_desc = [&](uint32_t step) {
        return sdesc_noswz(smem_u32(smem + C::kOffStats + (step % C::kQBufs) * kStatsTileBytes), 128, 256);
      };
      auto issue_fold_s = [&](uint32_t step) { umma_ss(tmem + C::kTmST, a_lse, stats_desc(step), idesc_s, 1u); };
      auto issue_fold_dp = [&](uint32_t step) { umma_ss(tmem + C::kTmDPT, a_d, stats_desc(step), idesc_s, 1u); };
      // Short d = 64 tiles take the next tile during the last step and may issue its first
      // scores there; long tiles and d = 128 keep the plain loop (the restructured one
      // measured 2-3 % slower on long tiles, where a tile boundary is rare).
      if constexpr (kAhead) {
        uint32_t s = 0;
        int it = 0;
        bool ok = true;
        int tile = take_tile(0, 0x50f);
        bool first_issued = false;   // this tile's first scores went out during the previous tile's last step
        for (;; ++it) {
          if (tile < 0) break;
          int kb, bh;
          group_order(tile, BHkv, nb, hg, kb, bh);
          const int kvb = it % C::kKVBufs;
          const int q0 = CAUSAL ? kb : 0;
          const int nsteps = SPARSE ? sparse_n(kb) : group * (nb - q0);
          if (!wait_warp(bar(C::kKVFull + kvb), (it / C::kKVBufs) & 1, ctl, 0x501)) break;
          const uint32_t kbase = smem_u32(smem + C::kOffK + kvb * C::kTileBytes);
          const uint32_t vbase = smem_u32(smem + C::kOffV + kvb * C::kTileBytes);
          // first block of the tile
          if (!first_issued) {
            if (!wait_warp(bar(C::kQFull + s % C::kQBufs), (s / C::kQBufs) & 1, ctl, 0x502) ||
                (s > 0 && !wait_warp(bar(C::kSTFree), (s - 1) & 1, ctl, 0x503)) ||
                (!C::kEarly && s > 0 && !wait_warp(bar(C::kDQFree), (s - 1) & 1, ctl, 0x504))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              issue_st(kbase, qaddr(s));
              issue_fold_s(s);
              issue_dpt(vbase, oaddr(s));
              issue_fold_dp(s);
              umma_commit(bar(C::kSFull));
            }
            __syncwarp();
          }
          first_issued = false;
          int next_tile = -2;   // taken during the last step
          for (int i = 0; i < nsteps; ++i, ++s) {
            const bool last = (i == nsteps - 1);
            if (kAhead && last) {
              // the next tile's first S^T and dP^T now, ahead of this block's gradients, when its
              // K/V and first Q/dO have landed (the producer loaded them a tile ahead)
              next_tile = take_tile(it + 1, 0x50e);
              if (next_tile >= 0) {
                const int kvn = (it + 1) % C::kKVBufs;
                const bool ready =
                    __all_sync(0xffffffffu, mbar_test(bar(C::kKVFull + kvn), ((it + 1) / C::kKVBufs) & 1) != 0u &&
                                                mbar_test(bar(C::kQFull + (s + 1) % C::kQBufs),
                                                              ((s + 1) / C::kQBufs) & 1) != 0u);
                if (ready) {
                  if (!wait_warp(bar(C::kSTFree), s & 1, ctl, 0x50d)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  if (elect_one()) {
                    issue_st(smem_u32(smem + C::kOffK + kvn * C::kTileBytes), qaddr(s + 1));
                    issue_fold_s(s + 1);
                    issue_dpt(smem_u32(smem + C::kOffV + kvn * C::kTileBytes), oaddr(s + 1));
                    issue_fold_dp(s + 1);
                    umma_commit(bar(C::kSFull));
                  }
                  __syncwarp();
                  first_issued = true;
                }
              }
            }
            if (C::kEarly && !last) {
              if (!wait_warp(bar(C::kQFull + (s + 1) % C::kQBufs), ((s + 1) / C::kQBufs) & 1, ctl, 0x505) ||
                  !wait_warp(bar(C::kSTFree), s & 1, ctl, 0x506)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_st(kbase, qaddr(s + 1));
                issue_fold_s(s + 1);
                issue_dpt(vbase, oaddr(s + 1));
                issue_fold_dp(s + 1);
                umma_commit(bar(C::kSFull));
              }
              __syncwarp();
            }
            if (!wait_warp(bar(C::kDSFull), s & 1, ctl, 0x507) ||
                (i == 0 && it > 0 && !wait_warp(bar(C::kDKVEmpty), (it - 1) & 1, ctl, 0x508))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              const uint32_t qbase = qaddr(s), obase = oaddr(s);
              const uint64_t dsk = sdesc_sw128(dst, 16, 1024);                 // dS^T, K-major (A of dK)
              const uint64_t omn = sdesc_sw128(obase, kChunkBytes, 1024);      // dO, MN-major (B of dV)
              const uint64_t qmn = sdesc_sw128(qbase, kChunkBytes, 1024);      // Q, MN-major (B of dK)
  #pragma unroll
              for (int kk = 0; kk < kRows / 16; ++kk) {
                const uint32_t acc = (i == 0 && kk == 0) ? 0u : 1u;
                const uint32_t rows16 = (kk * 16 * 128) >> 4;                  // 16 rows of 128 bytes
                // dV += P^T dO: A = P^T from tensor memory (16 query columns = 8 packed columns)
                umma_ts(tmem + C::kTmDV, tmem + C::tm_pt(kk >> 2) + (kk & 3) * 8, omn + rows16, idesc_kv, acc);
                // dK += dS^T Q: A = dS^T (keys x q, q contiguous), K-major, 16 q = 32 bytes
                const uint32_t aoff = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                umma_ss(tmem + C::kTmDK, dsk + aoff, qmn + rows16, idesc_kv, acc);
              }
              // d = 128 (one Q/dO buffer): dV and dK are the last readers of this block's Q
              // and dO, so the producer may refill the buffer while dQ (which reads dS and K)
              // still runs.  (At d = 64, with three buffers, the earlier refill only competes
              // with dQ and measured slower.)
              if constexpr (!C::kEarly) umma_commit(bar(C::kQEmpty + s % C::kQBufs));
              // d = 64: dK and dV are final after the tile's last dV and dK products: hand their
              // columns to the read-out now, not after the last dQ product
              if (kAhead && last) umma_commit(bar(C::kDKVFull));
            }
            __syncwarp();
            // d = 64: dQ has its own columns, which the dQ warpgroup must have read out for
            // the previous block; dV and dK above did not wait for that (at a tile's first
            // block the same warpgroup is also writing the previous tile's dK and dV)
            if (C::kEarly && s > 0 && !wait_warp(bar(C::kDQFree), (s - 1) & 1, ctl, 0x509)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              const uint64_t dsmn = sdesc_sw128(dst, kChunkBytes, 1024);       // dS, MN-major (A of dQ)
              const uint64_t kmn = sdesc_sw128(kbase, kChunkBytes, 1024);      // K, MN-major (B of dQ)
  #pragma unroll
              for (int kk = 0; kk < kRows / 16; ++kk) {
                // dQ = dS K: A = dS (q x keys) read MN-major from the dS^T block; B = K MN-major
                const uint32_t rows16 = (kk * 16 * 128) >> 4;
                umma_ss(tmem + C::kTmDQ, dsmn + rows16, kmn + rows16, idesc_q, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(C::kMmaDone));
              if constexpr (C::kEarly) umma_commit(bar(C::kQEmpty + s % C::kQBufs));
              umma_commit(bar(C::kDQFull));
            }
            __syncwarp();
            if (!C::kEarly && !last) {
              // S^T(next) overwrites the S^T columns that P^T(this) shared; tcgen05.mma
              // from one thread run in issue order, so dV above has read P^T first.
              if (!wait_warp(bar(C::kQFull + (s + 1) % C::kQBufs), ((s + 1) / C::kQBufs) & 1, ctl, 0x50a) ||
                  !wait_warp(bar(C::kSTFree), s & 1, ctl, 0x50b)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_st(kbase, qaddr(s + 1));
                issue_fold_s(s + 1);
              }
              __syncwarp();
              // dP^T(next) overwrites the dP^T columns that dQ(this) occupies
              if (!wait_warp(bar(C::kDQFree), s & 1, ctl, 0x50c)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_dpt(vbase, oaddr(s + 1));
                issue_fold_dp(s + 1);
                umma_commit(bar(C::kSFull));
              }
              __syncwarp();
            }
          }
          if (!ok) break;
          if (elect_one()) {
            umma_commit(bar(C::kKVEmpty + kvb));
            if constexpr (!kAhead) umma_commit(bar(C::kDKVFull));
          }
          __syncwarp();
          tile = next_tile != -2 ? next_tile : take_tile(it + 1, 0x50f);
        }
      } else {
        uint32_t s = 0;
        int it = 0;
        bool ok = true;
        for (;; ++it) {
          const int tile = take_tile(it, 0x50f);
          if (tile < 0) break;
          int kb, bh;
          group_order(tile, BHkv, nb, hg, kb, bh);
          const int kvb = it % C::kKVBufs;
          const int q0 = CAUSAL ? kb : 0;
          const int nsteps = SPARSE ? sparse_n(kb) : group * (nb - q0);
          if (!wait_warp(bar(C::kKVFull + kvb), (it / C::kKVBufs) & 1, ctl, 0x501)) break;
          const uint32_t kbase = smem_u32(smem + C::kOffK + kvb * C::kTileBytes);
          const uint32_t vbase = smem_u32(smem + C::kOffV + kvb * C::kTileBytes);
          // first block of the tile
          if (!wait_warp(bar(C::kQFull + s % C::kQBufs), (s / C::kQBufs) & 1, ctl, 0x502) ||
              (s > 0 && !wait_warp(bar(C::kSTFree), (s - 1) & 1, ctl, 0x503)) ||
              (!C::kEarly && s > 0 && !wait_warp(bar(C::kDQFree), (s - 1) & 1, ctl, 0x504))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_st(kbase, qaddr(s));
            issue_fold_s(s);
            issue_dpt(vbase, oaddr(s));
            issue_fold_dp(s);
            umma_commit(bar(C::kSFull));
          }
          __syncwarp();
          for (int i = 0; i < nsteps; ++i, ++s) {
            const bool last = (i == nsteps - 1);
            if (C::kEarly && !last) {
              if (!wait_warp(bar(C::kQFull + (s + 1) % C::kQBufs), ((s + 1) / C::kQBufs) & 1, ctl, 0x505) ||
                  !wait_warp(bar(C::kSTFree), s & 1, ctl, 0x506)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_st(kbase, qaddr(s + 1));
                issue_fold_s(s + 1);
                issue_dpt(vbase, oaddr(s + 1));
                issue_fold_dp(s + 1);
                umma_commit(bar(C::kSFull));
              }
              __syncwarp();
            }
            if (!wait_warp(bar(C::kDSFull), s & 1, ctl, 0x507) ||
                (i == 0 && it > 0 && !wait_warp(bar(C::kDKVEmpty), (it - 1) & 1, ctl, 0x508))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              const uint32_t qbase = qaddr(s), obase = oaddr(s);
              const uint64_t dsk = sdesc_sw128(dst, 16, 1024);                 // dS^T, K-major (A of dK)
              const uint64_t omn = sdesc_sw128(obase, kChunkBytes, 1024);      // dO, MN-major (B of dV)
              const uint64_t qmn = sdesc_sw128(qbase, kChunkBytes, 1024);      // Q, MN-major (B of dK)
  #pragma unroll
              for (int kk = 0; kk < kRows / 16; ++kk) {
                const uint32_t acc = (i == 0 && kk == 0) ? 0u : 1u;
                const uint32_t rows16 = (kk * 16 * 128) >> 4;                  // 16 rows of 128 bytes
                // dV += P^T dO: A = P^T from tensor memory (16 query columns = 8 packed columns)
                umma_ts(tmem + C::kTmDV, tmem + C::tm_pt(kk >> 2) + (kk & 3) * 8, omn + rows16, idesc_kv, acc);
                // dK += dS^T Q: A = dS^T (keys x q, q contiguous), K-major, 16 q = 32 bytes
                const uint32_t aoff = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                umma_ss(tmem + C::kTmDK, dsk + aoff, qmn + rows16, idesc_kv, acc);
              }
              // d = 128 (one Q/dO buffer): dV and dK are the last readers of this block's Q
              // and dO, so the producer may refill the buffer while dQ (which reads dS and K)
              // still runs.  (At d = 64, with three buffers, the earlier refill only competes
              // with dQ and measured slower.)
              if constexpr (!C::kEarly) umma_commit(bar(C::kQEmpty + s % C::kQBufs));
            }
            __syncwarp();
            // d = 64: dQ has its own columns, which the dQ warpgroup must have read out for
            // the previous block; dV and dK above did not wait for that (at a tile's first
            // block the same warpgroup is also writing the previous tile's dK and dV)
            if (C::kEarly && s > 0 && !wait_warp(bar(C::kDQFree), (s - 1) & 1, ctl, 0x509)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              const uint64_t dsmn = sdesc_sw128(dst, kChunkBytes, 1024);       // dS, MN-major (A of dQ)
              const uint64_t kmn = sdesc_sw128(kbase, kChunkBytes, 1024);      // K, MN-major (B of dQ)
  #pragma unroll
              for (int kk = 0; kk < kRows / 16; ++kk) {
                // dQ = dS K: A = dS (q x keys) read MN-major from the dS^T block; B = K MN-major
                const uint32_t rows16 = (kk * 16 * 128) >> 4;
                umma_ss(tmem + C::kTmDQ, dsmn + rows16, kmn + rows16, idesc_q, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(C::kMmaDone));
              if constexpr (C::kEarly) umma_commit(bar(C::kQEmpty + s % C::kQBufs));
              umma_commit(bar(C::kDQFull));
            }
            __syncwarp();
            if (!C::kEarly && !last) {
              // S^T(next) overwrites the S^T columns that P^T(this) shared; tcgen05.mma
              // from one thread run in issue order, so dV above has read P^T first.
              if (!wait_warp(bar(C::kQFull + (s + 1) % C::kQBufs), ((s + 1) / C::kQBufs) & 1, ctl, 0x50a) ||
                  !wait_warp(bar(C::kSTFree), s & 1, ctl, 0x50b)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_st(kbase, qaddr(s + 1));
                issue_fold_s(s + 1);
              }
              __syncwarp();
              // dP^T(next) overwrites the dP^T columns that dQ(this) occupies
              if (!wait_warp(bar(C::kDQFree), s & 1, ctl, 0x50c)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_dpt(vbase, oaddr(s + 1));
                issue_fold_dp(s + 1);
                umma_commit(bar(C::kSFull));
              }
              __syncwarp();
            }
          }
          if (!ok) break;
          if (elect_one()) {
            umma_commit(bar(C::kKVEmpty + kvb));
            umma_commit(bar(C::kDKVFull));
          }
          __syncwarp();
        }
      }
      if (elect_one()) umma_commit(bar(C::kDrain));
      __syncwarp();
      mbar_wait(bar(C::kDrain), 0, drain, 0x5f1);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ dS warpgroups
    regs_inc<kDsRegs>();
    const int h = warp >> 2;                     // query half
    const int t = threadIdx.x & 127;             // key row inside the block
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t st_addr = tmem + lane_base + C::kTmST + 64 * h;
    const uint32_t dpt_addr = tmem + lane_base + C::kTmDPT + 64 * h;
    const uint32_t pt_addr = tmem + lane_base + C::tm_pt(h);
    uint8_t* dst_chunk = smem + C::kOffDST + h * kChunkBytes;
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    uint32_t s = 0;
    for (int k = 0;; ++k) {
      const int tile = take_tile(k, 0x60f);
      if (tile < 0) break;
      int kb, bh;
      group_order(tile, BHkv, nb, hg, kb, bh);
      const int q0 = SPARSE ? sparse_q(kb, 0) : (CAUSAL ? kb : 0);
      const int nq = SPARSE ? sparse_n(kb) : 0;
      bool ok = true;
      for (int g = 0; ok && g < group; ++g)
      for (int qi = q0, j = 0; SPARSE ? j < nq : qi < nb; ++s, ++j, qi = SPARSE ? sparse_q(kb, j) : qi + 1) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kSFull), s & 1, ctl, 0x601))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64], pr[64];
        tmem_ld32(st_addr, sr);
        tmem_ld32(st_addr + 32, sr + 32);
        tmem_ld32(dpt_addr, pr);
        tmem_ld32(dpt_addr + 32, pr + 32);
        tmem_ld_wait();
        reg_fence<64>(sr);
        reg_fence<64>(pr);
        tc_fence_before();
        mbar_arrive(bar(C::kSTFree));
        if (CAUSAL && qi == kb) {   // key t is visible to query column c iff t <= c: P = 0 elsewhere
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (64 * h + e < t) sr[e] = 0xFF800000u;   // -inf: 2^-inf = 0, and dS = 0 * (dP - D) = 0
        }
        uint32_t pw[32], dw[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {   // two query columns at a time
          // the tensor memory holds S^T - lse/scale and dP^T - D already
          float x0, x1;
          f2_unpack(fmul2(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          float d0, d1;
          f2_unpack(fmul2(f2_pack(p0, p1), f2_pack(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1]))), d0, d1);
          pw[e >> 1] = pack2<DT>(p0, p1);
          dw[e >> 1] = pack2<DT>(d0, d1);
        }
        // the previous block's gradient MMAs must be done with P^T and dS^T
        if (!__all_sync(0xffffffffu, s == 0 || mbar_wait(bar(C::kMmaDone), (s - 1) & 1, ctl, 0x603))) {
          ok = false;
          break;
        }
        tmem_st32(pt_addr, pw);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(dst_chunk + sw128_offset(t, u)) =
              make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kDSFull));
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup: dQ reduction, dK/dV epilogue
    regs_dec<kDqRegs<D>>();
    const int u = threadIdx.x - 256;
    const int dq_warp = warp - 8;          // rows 32*dq_warp .. +31 of each query block
    const int lane = threadIdx.x & 31;
    uint32_t dq_chunks = 0;                // chunks this warp has staged (its ring position)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // dK (times scale) and dV of the key block, read out of tensor memory; the columns
    // are handed back to the MMA warp as soon as the last of them is in registers.  Each
    // warp stages its 32 rows as 16-bit values in its own dQ staging ring (4 KB per 64
    // columns, 128-byte swizzle: conflict-free) and writes them with bulk tensor stores,
    // instead of one 16-byte global store per row and unit (32 lines per instruction)
    bool dkdv_staged = false;   // the ring holds dK/dV rows that a store may still be reading
    auto write_dkdv_staged = [&](int it, int kb, int bh) -> bool {
      if (!wait_warp(bar(C::kDKVFull), it & 1, ctl, 0x702)) return false;
      tc_fence_after();
      uint8_t* ring = smem + C::kOffDQS + dq_warp * C::kDQRing * C::kDQChunkBytes;
      const int row0 = kb * kRows + 32 * dq_warp;   // rows past N are not written by the store
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = which == 0 ? C::kTmDV : C::kTmDK;
        const float mul = which == 0 ? 1.0f : scale;
        // every earlier bulk operation of this warp (dQ reductions, the dV store) has read the ring
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + col0 + c * 32, r);
          tmem_ld_wait();
          reg_fence<32>(r);
          if (which == 1 && c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::kDKVEmpty));
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack2<DT>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
          // 32 columns are 4 of the 8 16-byte units of this lane's 128-byte row in block c / 2
          uint8_t* row = ring + (c >> 1) * 4096 + lane * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(row + ((((c & 1) * 4 + v) ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int c2 = 0; c2 < D / 64; ++c2)
            tma_store_3d(which == 0 ? &tm_dv : &tm_dk, smem_u32(ring) + c2 * 4096, c2 * 64, row0, bh);
          bulk_commit_group();
        }
      }
      dkdv_staged = true;
      return true;
    };
    // (long tiles and d = 128: one 16-byte global store per row and unit, measured
    // faster there than the staged form above)
    auto write_dkdv_rows = [&](int it, int kb, int bh) -> bool {
      if (!wait_warp(bar(C::kDKVFull), it & 1, ctl, 0x702)) return false;
      tc_fence_after();
      const int key = kb * kRows + u;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = which == 0 ? C::kTmDV : C::kTmDK;
        const float mul = which == 0 ? 1.0f : scale;
        uint8_t* grow = reinterpret_cast<uint8_t*>(which == 0 ? dv : dk) + ((size_t)bh * N + key) * (D * 2);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + col0 + c * 32, r);
          tmem_ld_wait();
          reg_fence<32>(r);
          if (which == 1 && c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::kDKVEmpty));
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack2<DT>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
          if (key < N) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              st_global_v4(grow + c * 64 + i * 16, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
      return true;
    };
    auto write_dkdv = [&](int it, int kb, int bh) -> bool {
      if constexpr (kStagedDKV) return write_dkdv_staged(it, kb, bh);
      else return write_dkdv_rows(it, kb, bh);
    };
    uint32_t s = 0;
    int it = 0;
    for (;; ++it) {
      const int tile = take_tile(it, 0x70f);
      if (tile < 0) break;
      int kb, bh;
      group_order(tile, BHkv, nb, hg, kb, bh);
      const int q0 = SPARSE ? sparse_q(kb, 0) : (CAUSAL ? kb : 0);
      const int nq = SPARSE ? sparse_n(kb) : 0;
      bool ok = true;
      for (int g = 0; ok && g < group; ++g) {
      const int bhq = first_q_head(bh) + g;
      for (int qi = q0, j = 0; SPARSE ? j < nq : qi < nb; ++s, ++j, qi = SPARSE ? sparse_q(kb, j) : qi + 1) {
        const bool tile_last = g == group - 1 && (SPARSE ? j == nq - 1 : qi == nb - 1);
        // short d = 64 tiles: dK and dV are handed over after the tile's last dV and dK
        // products, before its last dQ product: they are read out first
        if (kAhead && tile_last && !write_dkdv(it, kb, bh)) {
          ok = false;
          break;
        }
        if (!wait_warp(bar(C::kDQFull), s & 1, ctl, 0x701)) {
          ok = false;
          break;
        }
        // long d = 64 tiles: the next tile's first gradient MMAs wait for the dK/dV columns,
        // so those are read out before the last dQ of the tile (at d = 128 the next tile's
        // first scores wait for the dQ columns instead, so dQ goes first)
        if (C::kEarly && !kAhead && tile_last && !write_dkdv(it, kb, bh)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < D / 64; ++half) {   // 64 columns per staging round
          uint32_t r[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld32(tmem + lane_base + C::kTmDQ + half * 64 + c * 32, r[c]);
          tmem_ld_wait();
          reg_fence<32>(r[0]);
          reg_fence<32>(r[1]);
          if (half == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::kDQFree));
          }
#pragma unroll
          for (int q = 0; q < 64 / C::kDQCols; ++q) {   // chunks of kDQCols columns
            uint8_t* box = smem + C::kOffDQS + (dq_warp * C::kDQRing + dq_chunks % C::kDQRing) * C::kDQChunkBytes;
            // the reduction that last read this buffer must be done reading it (after a
            // dK/dV write-out: the stores, which read the whole ring)
            if (lane == 0) {
              if (dkdv_staged) bulk_wait_read<0>();
              else if (dq_chunks >= (uint32_t)C::kDQRing) bulk_wait_read<C::kDQRing - 1>();
            }
            __syncwarp();
            dkdv_staged = false;
            if constexpr (WIDE) {
              const uint32_t* src = r[q];
#pragma unroll
              for (int v = 0; v < 8; ++v)   // 128-byte rows, 16-byte units swizzled by row mod 8
                *reinterpret_cast<uint4*>(box + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                    make_uint4(src[4 * v], src[4 * v + 1], src[4 * v + 2], src[4 * v + 3]);
            } else {
              const uint32_t* src = r[q >> 1] + (q & 1) * 16;
#pragma unroll
              for (int v = 0; v < 4; ++v)   // 64-byte rows, 16-byte units swizzled by (row / 2) mod 4
                *reinterpret_cast<uint4*>(box + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(src[4 * v], src[4 * v + 1], src[4 * v + 2], src[4 * v + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_3d(&tm_dq, smem_u32(box), half * 64 + q * C::kDQCols, qi * kRows + 32 * dq_warp, bhq);
              bulk_commit_group();
            }
            ++dq_chunks;
          }
        }
      }
      }
      if (!ok) break;
      if (!C::kEarly && !write_dkdv(it, kb, bh)) break;
    }
    // every bulk reduction issued by this warp must complete before the CTA exits
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// x as three 16-bit terms, x = 256 h + m + l to about 24 significant bits: h = x/256
// rounded, m = the remainder rounded, l = what is left rounded (each remainder is exact in
// float32).  One 16-byte core-matrix row: (h, m, l, 0, 0, 0, 0, 0).
template <int DT>
__device__ __forceinline__ uint4 split3(float x) {
  const uint32_t h = pack2<DT>(x * (1.0f / 256.0f), 0.0f) & 0xFFFFu;
  const float r1 = x - 256.0f * unpack2<DT>(h).x;
  const uint32_t m = pack2<DT>(r1, 0.0f) & 0xFFFFu;
  const uint32_t l = pack2<DT>(r1 - unpack2<DT>(m).x, 0.0f) & 0xFFFFu;
  return make_uint4(h | (m << 16), l, 0u, 0u);
}

// Per query row: -lse/scale and -D = -rowsum(dO o O), written in three 16-bit terms each
// into the row's line of its block's statistics tile (kStatsTileBytes layout); padding
// rows get zeros (their Q and dO rows read as zero, so they add nothing whatever P is).
// Also zeroes the float32 dQ accumulator and the tile counter.  D/8 threads per row
// (8 for d = 64, 16 for d = 128), each reading 16 bytes of O and of dO.
template <int D, int DT>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                      const float* __restrict__ lse, uint8_t* __restrict__ stats,
                                                      float* __restrict__ dq_accum,
                                                      unsigned int* __restrict__ tile_counter, int BH, int N, int Npad,
                                                      float inv_scale, size_t accum_elems) {
  constexpr int kTPR = D / 8;   // threads per row
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gtid / kTPR;  // padded row index over BH*Npad
  const int part = (int)(gtid % kTPR);
  const long long rows = (long long)BH * Npad;
  grid_dep_wait();
  grid_dep_launch();
  if (gtid == 0) *tile_counter = 0u;
  const int bh = (int)(row / Npad);
  const int n = (int)(row - (long long)bh * Npad);
  float acc = 0.f;
  const bool valid = (row < rows) && (n < N);
  if (valid) {
    const size_t base = ((size_t)bh * N + n) * D + part * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + base);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + base);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa = unpack2<DT>(aw[i]);
      const float2 fb = unpack2<DT>(bw[i]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int off = kTPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0 && row < rows) {
    const float nl = valid ? -lse[(size_t)bh * N + n] * inv_scale : 0.f;
    const float nd = valid ? -acc : 0.f;
    uint8_t* line = stats + (size_t)(row >> 7) * kStatsTileBytes + ((row & 127) >> 3) * 256 + (row & 7) * 16;
    *reinterpret_cast<uint4*>(line) = split3<DT>(nl);
    *reinterpret_cast<uint4*>(line + 128) = split3<DT>(nd);
  }
  // zero the accumulator (grid-stride, 16 bytes per thread per step)
  const size_t n4 = accum_elems / 4;
  for (size_t i = (size_t)gtid; i < n4; i += (size_t)gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(dq_accum)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dq = scale * dq_accum, rounded to the 16-bit type; 8 elements per thread.
template <int DT>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                     float scale, size_t n8) {
  grid_dep_wait();
  grid_dep_launch();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 w;
    w.x = pack2<DT>(a.x * scale, a.y * scale);
    w.y = pack2<DT>(a.z * scale, a.w * scale);
    w.z = pack2<DT>(b.x * scale, b.y * scale);
    w.w = pack2<DT>(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = w;
  }
}

template <int D, int DT, bool CAUSAL, int MODE, bool WIDE>
cudaError_t launch_kv_t(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D, WIDE>;
  auto kern = bwd_kv_kernel<D, DT, CAUSAL, MODE, WIDE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // the setmaxnreg split inside the kernel must fit what the launch provides
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kBwdThreads < (2 * kDsRegs + kDqRegs<D> + kCtlRegs<D>) * 128) return cudaErrorInvalidConfiguration;
  const int nb = (a.N + kRows - 1) / kRows;
  const int ntiles = a.BHkv * nb;
  const int grid = ntiles < a.num_sms ? ntiles : a.num_sms;
  return launch_overlapped(kern, grid, kBwdThreads, C::kSmemBytes, stream, a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dq,
                           a.tm_dk, a.tm_dv, a.stats, a.dq_accum, a.tile_counter, static_cast<uint16_t*>(a.dk),
                           static_cast<uint16_t*>(a.dv), a.BHkv, a.H, a.G, a.N, a.Npad, a.scale, a.scale_log2,
                           a.heads_per_group, a.err_word, a.limit_ns);
}

template <int D, int DT, bool CAUSAL, int MODE>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream, int stages) {
  if (stages & kBwdStagePre) {
    constexpr int kTPR = D / 8;
    const long long threads = (long long)a.BH * a.Npad * kTPR;
    long long blocks = (threads + 255) / 256;
    const long long min_blocks = 4LL * a.num_sms;   // enough blocks to zero the accumulator quickly
    if (blocks < min_blocks) blocks = min_blocks;
    const size_t accum_elems = (size_t)a.BH * a.N * D;
    cudaError_t e = launch_overlapped(bwd_pre_kernel<D, DT>, (unsigned)blocks, 256, 0, stream,
                                      static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dO), a.lse,
                                      a.stats, a.dq_accum, a.tile_counter, a.BH, a.N, a.Npad, 1.0f / a.scale,
                                      accum_elems);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageKV) {
    cudaError_t e;
    if constexpr (D == 64 && MODE == 0)
      e = a.wide_dq ? launch_kv_t<D, DT, CAUSAL, MODE, true>(a, stream) : launch_kv_t<D, DT, CAUSAL, MODE, false>(a, stream);
    else
      e = launch_kv_t<D, DT, CAUSAL, MODE, false>(a, stream);
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdStageDQ) {
    const size_t n8 = (size_t)a.BH * a.N * D / 8;
    long long blocks = (long long)((n8 + 255) / 256);
    if (blocks > 8LL * a.num_sms) blocks = 8LL * a.num_sms;
    if (blocks < 1) blocks = 1;
    return launch_overlapped(bwd_dq_kernel<DT>, (unsigned)blocks, 256, 0, stream, a.dq_accum,
                             static_cast<uint16_t*>(a.dq), a.scale, n8);
  }
  return cudaSuccess;
}

template <int MODE>
cudaError_t launch_bwd_g(const BwdArgs& a, cudaStream_t stream, int stages) {
  const int key = (a.d == 128 ? 4 : 0) | (a.dtype == 1 ? 2 : 0) | (a.causal ? 1 : 0);
  switch (key) {
    case 0: return launch_bwd_t<64, 0, false, MODE>(a, stream, stages);
    case 1: return launch_bwd_t<64, 0, true, MODE>(a, stream, stages);
    case 2: return launch_bwd_t<64, 1, false, MODE>(a, stream, stages);
    case 3: return launch_bwd_t<64, 1, true, MODE>(a, stream, stages);
    case 4: return launch_bwd_t<128, 0, false, MODE>(a, stream, stages);
    case 5: return launch_bwd_t<128, 0, true, MODE>(a, stream, stages);
    case 6: return launch_bwd_t<128, 1, false, MODE>(a, stream, stages);
    default: return launch_bwd_t<128, 1, true, MODE>(a, stream, stages);
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int stages) {
  if (a.pattern == 1) return launch_bwd_g<2>(a, stream, stages);
  return a.G != 1 ? launch_bwd_g<1>(a, stream, stages) : launch_bwd_g<0>(a, stream, stages);
}

}  // namespace fa
