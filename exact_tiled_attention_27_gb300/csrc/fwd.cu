// fwd.cu -- forward kernel of exact tiled attention for sm_103a.
//
// One persistent CTA per SM walks work tiles, heaviest causal tiles first.  A work
// tile is one (batch*head) and two adjacent 128-row query blocks ("sub-tiles" 0 and
// 1) that share every K/V block loaded for them.  Inside a CTA the work is split by
// role:
//
//   warps 0-3   softmax warpgroup of sub-tile 0 (one thread per query row)
//   warps 4-7   softmax warpgroup of sub-tile 1
//   warp 8      TMA producer: the Q pair, then a ring of K/V stages
//   warp 9      MMA issuer (one thread): S_t = Q_t K^T into tensor memory and
//               O_t += P_t V with P_t read from tensor memory, alternating between
//               the two sub-tiles so that one sub-tile's softmax overlaps the other
//               sub-tile's matrix products
//
// A softmax thread reads its row of S from tensor memory, masks the causal diagonal
// and the ragged tail, updates the running maximum m and running sum l, rescales its
// row of the unnormalised O when m moved, writes P (16-bit) back to tensor memory,
// and in the epilogue divides O by l and stores O and lse.
//
// The method follows the "Flash Attention" chapter (mlx.void.app): section
// "地基：流式 softmax" for the running (m, l) and the e^{m_old-m_new} patch,
// "FlashAttention——把整件事分块塞进 SRAM" for the query-outer / key-value-inner tiling in
// which the score tile never leaves the chip, and "FlashAttention-2" for the
// deferred division by l, the splitting of the sequence into query blocks across
// the whole chip, and the skipping of tiles wholly above the causal diagonal.
// Exponentials are taken in base 2 with scale*log2(e) folded into one FMA.
//
// Ordering facts the pipeline relies on:
//  * every sub-tile has one S buffer; the MMA thread issues S_t(j+1) after
//    O_t += P_t(j) V(j) and commits both to one barrier, so when the softmax sees
//    S_t(j+1) the previous P.V has already landed in O_t and O_t can be rescaled
//    without any further wait;
//  * tcgen05.mma operations issued by one thread execute in issue order (P_t occupies
//    the first 64 columns of S_t's buffer, and S_t(j+1) is issued after P_t(j).V).
//
// O is divided by the sum of the 16-bit P values the P.V product actually used, so
// each output row is an exact convex combination of V rows with those weights and
// the rounding of a dominant weight cancels; lse uses the sum of the unrounded P.
// At d = 64 the tensor core forms that sum (a block of ones as 16 more V columns);
// at d = 128 the softmax threads add it up.
//
// The running maximum is only moved when a new row maximum exceeds it by more than a
// threshold T (base-2 units).  Until then P entries may reach 2^T; the result is
// unchanged because l and O are accumulated against the same maximum, and the O rescale
// is skipped on most blocks.  T is as large as the 16-bit P allows with margin: 15 for
// fp16 (largest finite 65504 > 2^15), 32 for bf16 (whose range is float32's; O and l,
// float32, stay below 2^(32 + 31) times |V|).  With scores of standard deviation 13
// (base 2), T = 8 rescaled some row of a warp on 46 % of the blocks, T = 32 on 0.4 %.
#include <cuda_fp16.h>

#include <algorithm>
#include <vector>

#include "fwd_tiles.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;    // 2 softmax warpgroups + (producer, MMA, 2 idle) warpgroup
// Register split: the kernel is compiled for kLaunchRegs per thread; the third
// warpgroup gives registers back so the softmax warpgroups can hold a whole row of S.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 216;
constexpr int kOtherRegs = 64;
static_assert((2 * kSoftmaxRegs + kOtherRegs) * 128 <= kLaunchRegs * kThreads, "register split exceeds the launch");
constexpr int kChunkBytes = kTileRows * 128;   // one 128-row x 128-byte swizzle column block
template <int DT>
constexpr float kRescaleThreshold = DT == 1 ? 15.0f : 32.0f;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;                    // 64 16-bit elements per 128-byte row
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kQBufs = (D == 64) ? 2 : 1;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kOffQ = 0;                           // [kQBufs][2 sub-tiles]
  static constexpr int kOffK = kOffQ + kQBufs * 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  // d = 64: a 128-row block of ones forms 16 extra columns of V, so P.V also yields
  // the sum of the 16-bit P values (O column 64); d = 128 has no tensor-memory columns
  // to spare and sums them on the CUDA cores instead.
  static constexpr bool kOnesCol = (D == 64);
  static constexpr int kOffOnes = kOffV + kStages * kTileBytes;
  // split tiles: sub-tile 1's running maximum and sum per row, for sub-tile 0's merge
  static constexpr int kOffMerge = kOffOnes + (kOnesCol ? kChunkBytes : 0);
  static constexpr int kOffBar = kOffMerge + 2 * kTileRows * 4;
  static constexpr uint32_t kPVN = D + (kOnesCol ? 16 : 0);   // N of the P.V MMA
  // barrier indices
  static constexpr int kQFull = 0;                          // [kQBufs]
  static constexpr int kQEmpty = kQFull + kQBufs;           // [kQBufs]
  static constexpr int kKFull = kQEmpty + kQBufs;           // [kStages]
  static constexpr int kVFull = kKFull + kStages;           // [kStages]
  static constexpr int kKVEmpty = kVFull + kStages;         // [kStages]
  static constexpr int kSFull = kKVEmpty + kStages;         // [2]
  static constexpr int kPHalf = kSFull + 2;                 // [2] first 64 keys of P written
  static constexpr int kPFull = kPHalf + 2;                 // [2]
  static constexpr int kOFull = kPFull + 2;                 // [2]
  static constexpr int kOEmpty = kOFull + 2;                // [2]
  static constexpr int kMerge = kOEmpty + 2;                // split tiles: sub-tile 1's (m, l) published
  static constexpr int kMergeFree = kMerge + 1;             // ... and read by sub-tile 0
  static constexpr int kDrain = kMergeFree + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;   // + alignment slack
  // tensor memory columns (512 allocated)
  __host__ __device__ static constexpr uint32_t tm_s(int t) { return t * 128; }
  // P_t occupies the first 64 columns of S_t; O_t (kPVN columns) follows the S buffers
  __host__ __device__ static constexpr uint32_t tm_p(int t) { return t * 128; }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256 + t * 128; }
};

// MODE 1 (GEN): Nq != Nk or grouped key/value heads (fa_fwd_cross).  MODE 2 (SPARSE):
// the butterfly block pattern (fa_fwd_sparse).  MODE 0: Nq = Nk, every query head has
// its own key/value head, and rows always see at least one key.
template <int D, int DT, bool CAUSAL, int MODE, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, uint16_t* __restrict__ out, float* __restrict__ lse,
               int BH, int H, int G, int Nq, int Nk, float scale_log2, int pairing, unsigned int* err_word,
               uint64_t limit_ns) {
  using C = FwdCfg<D>;
  constexpr bool GEN = MODE == 1;
  constexpr bool SPARSE = MODE == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so
  // that every access through it stays a shared-memory access (not a generic one)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  // warp index through a shuffle so the compiler can treat it (and every TMEM
  // address, descriptor and loop bound derived from it) as warp-uniform
  const int warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const int nqb = (Nq + kTileRows - 1) / kTileRows;
  // d = 64 with single-block tiles: each tile's key blocks are split between the two
  // sub-tiles, which merge their partial results at the end (pairing 3)
  constexpr bool kSplit = D == 64 && SPLIT;
  const int ntiles = forward_tiles(BH, nqb, pairing);
  // key block of step j of tile ti: j, or the j-th block of the pair's butterfly list
  auto key_block = [&](const TileInfo& ti, int j) {
    return SPARSE ? bfly_block(ti.qb0 >> 1, j, (nqb + 1) >> 1, CAUSAL ? -1 : 0, 0) : j;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kQBufs; ++i) {
      mbar_init(bar(C::kQFull + i), 1);
      mbar_init(bar(C::kQEmpty + i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kSFull + t), 1);
      mbar_init(bar(C::kPHalf + t), kTileRows);
      mbar_init(bar(C::kPFull + t), kTileRows);
      mbar_init(bar(C::kOFull + t), 1);
      mbar_init(bar(C::kOEmpty + t), kTileRows);
    }
    mbar_init(bar(C::kMerge), kTileRows);
    mbar_init(bar(C::kMergeFree), kTileRows);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bar(C::kKFull + i), 1);
      mbar_init(bar(C::kVFull + i), 1);
      mbar_init(bar(C::kKVEmpty + i), 1);
    }
    mbar_init(bar(C::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (C::kOnesCol) {
    // the block of ones read as V columns 64..127 (only 64..79 are used)
    const uint32_t one2 = (DT == 1) ? 0x3C003C00u : 0x3F803F80u;
    uint4* ones = reinterpret_cast<uint4*>(smem + C::kOffOnes);
    for (int i = threadIdx.x; i < kChunkBytes / 16; i += kThreads) ones[i] = make_uint4(one2, one2, one2, one2);
    fence_proxy_async_smem();
  }
  if (warp == 9) {
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
  // (Dependents are not released early: they start when this grid completes.)
  grid_dep_wait();

  if (warp >= 8) {
    regs_dec<kOtherRegs>();
  }
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (whole warp; one lane issues)
    {
      if (elect_one()) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
      }
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int k = 0, tile = persistent_tile(0); ok && tile < ntiles; tile = persistent_tile(++k), ++it) {
        const TileInfo ti = decode_tile<MODE>(tile, BH, H, G, Nq, Nk, CAUSAL, pairing);
        const int qbuf = it % C::kQBufs;
        if (it >= C::kQBufs && !wait_warp(bar(C::kQEmpty + qbuf), ((it / C::kQBufs) - 1) & 1, ctl, 0x101)) {
          ok = false;
          break;
        }
        const bool split = kSplit && ti.split;
        const int nsub = split ? 1 : (ti.n1 > 0 ? 2 : 1);   // split: one query block for both
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::kQFull + qbuf), nsub * C::kTileBytes);
          for (int t = 0; t < nsub; ++t) {
            const uint32_t qdst = smem_u32(smem + C::kOffQ + (qbuf * 2 + t) * C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(qdst + c * kChunkBytes, &tm_q, bar(C::kQFull + qbuf), c * 64,
                          (t == 0 ? ti.qb0 : ti.qb1) * kTileRows,
                          ti.bh);
          }
        }
        __syncwarp();
        // split tiles: the loads alternate between the sub-tiles (load 2j + t is sub-tile
        // t's j-th block; sub-tile 0 takes the last one when it has one block more)
        const int nload = split ? ti.n0 + ti.n1 : ti.nkv;
        for (int ld = 0; ld < nload; ++ld, ++g) {
          const int kb = split ? key_block(ti, ld >> 1) + ((ld & 1) ? ti.koff1 : 0) : key_block(ti, ld);
          const int st = g % C::kStages;
          if (g >= (uint32_t)C::kStages &&
              !wait_warp(bar(C::kKVEmpty + st), ((g / C::kStages) - 1) & 1, ctl, 0x102)) {
            ok = false;
            break;
          }
          const uint32_t kdst = smem_u32(smem + C::kOffK + st * C::kTileBytes);
          const uint32_t vdst = smem_u32(smem + C::kOffV + st * C::kTileBytes);
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(C::kKFull + st), C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(kdst + c * kChunkBytes, &tm_k, bar(C::kKFull + st), c * 64, kb * kTileRows, ti.kvh);
            mbar_arrive_expect_tx(bar(C::kVFull + st), C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(vdst + c * kChunkBytes, &tm_v, bar(C::kVFull + st), c * 64, kb * kTileRows, ti.kvh);
          }
          __syncwarp();
        }
      }
      // On abort, every copy already issued must land before the CTA exits.
      if (!ok) {
        for (int st = 0; st < C::kStages; ++st) {
          if (g > (uint32_t)st) {
            const uint32_t last = g - 1 - ((g - 1 - st) % C::kStages);   // last step that used stage st
            mbar_wait(bar(C::kKFull + st), (last / C::kStages) & 1, drain, 0x1f1);
            mbar_wait(bar(C::kVFull + st), (last / C::kStages) & 1, drain, 0x1f2);
          }
        }
        for (int b = 0; b < C::kQBufs; ++b) {
          if (it > b) {
            const int last = it - 1 - ((it - 1 - b) % C::kQBufs);
            mbar_wait(bar(C::kQFull + b), (last / C::kQBufs) & 1, drain, 0x1f3);
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (whole warp; one lane issues)
    {
      constexpr uint32_t ab = (DT == 0) ? 1u : 0u;   // instruction-descriptor code: bf16 = 1, fp16 = 0
      constexpr uint32_t idesc_qk = idesc_f16(ab, 0, 0, 128, 128);
      constexpr uint32_t idesc_pv = idesc_f16(ab, 0, 1, 128, C::kPVN);
      uint32_t g = 0;
      int it = 0;
      uint32_t c[2] = {0, 0};   // steps issued per sub-tile (S-full / P-full phases)
      uint32_t e[2] = {0, 0};   // epilogues per sub-tile (O-full / O-empty phases)
      bool ok = true;
      auto issue_s = [&](int t, uint32_t qbase, uint32_t kbase) {
        const uint64_t qd = sdesc_sw128(qbase, 16, 1024);
        const uint64_t kd = sdesc_sw128(kbase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // A = Q (rows x d), B = K (keys x d): both K-major; 16 elements = 32 bytes
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          umma_ss(tmem + C::tm_s(t), qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      for (int k = 0, tile = persistent_tile(0); ok && tile < ntiles; tile = persistent_tile(++k), ++it) {
        const TileInfo ti = decode_tile<MODE>(tile, BH, H, G, Nq, Nk, CAUSAL, pairing);
        const int n[2] = {ti.n0, ti.n1};
        const int qbuf = it % C::kQBufs;
        const uint32_t qbase0 = smem_u32(smem + C::kOffQ + (qbuf * 2) * C::kTileBytes);
        if (!wait_warp(bar(C::kQFull + qbuf), (it / C::kQBufs) & 1, ctl, 0x201)) break;
        if (GEN && ti.nkv == 0) {   // no query row of the tile sees a key: nothing to multiply
          if (elect_one()) umma_commit(bar(C::kQEmpty + qbuf));
          __syncwarp();
          continue;
        }
        if constexpr (kSplit) {
          // both sub-tiles multiply the tile's one Q block with their own key blocks;
          // load 2j + t of the tile is sub-tile t's j-th key block, in a stage of its own
          auto ld_of = [&](int t, int j) { return g + 2u * (uint32_t)j + (uint32_t)t; };
          for (int t = 0; t < 2 && ok; ++t)
            if (n[t] > 0 && !wait_warp(bar(C::kKFull + ld_of(t, 0) % C::kStages), (ld_of(t, 0) / C::kStages) & 1,
                                       ctl, 0x202))
              ok = false;
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
            for (int t = 0; t < 2; ++t) {
              if (n[t] == 0) continue;
              issue_s(t, qbase0, smem_u32(smem + C::kOffK + (ld_of(t, 0) % C::kStages) * C::kTileBytes));
              umma_commit(bar(C::kSFull + t));
            }
          }
          __syncwarp();
          for (int j = 0; ok && j < ti.nkv; ++j) {
            for (int t = 0; t < 2; ++t) {
              if (j >= n[t]) continue;
              const uint32_t gj = ld_of(t, j), gn = ld_of(t, j + 1);
              const int st = gj % C::kStages, stn = gn % C::kStages;
              const bool more = j + 1 < n[t];
              if ((more && !wait_warp(bar(C::kKFull + stn), (gn / C::kStages) & 1, ctl, 0x203)) ||
                  !wait_warp(bar(C::kVFull + st), (gj / C::kStages) & 1, ctl, 0x204) ||
                  !wait_warp(bar(C::kPHalf + t), c[t] & 1, ctl, 0x205) ||
                  (j == 0 && e[t] > 0 && !wait_warp(bar(C::kOEmpty + t), (e[t] - 1) & 1, ctl, 0x206))) {
                ok = false;
                break;
              }
              const uint32_t vbase = smem_u32(smem + C::kOffV + st * C::kTileBytes);
              const uint64_t vd = sdesc_sw128(vbase, smem_u32(smem + C::kOffOnes) - vbase, 1024);
              auto issue_pv = [&](int kk0, int kk1) {
#pragma unroll
                for (int kk = kk0; kk < kk1; ++kk)
                  umma_ts(tmem + C::tm_o(t), tmem + C::tm_p(t) + kk * 8, vd + ((kk * 16 * 128) >> 4), idesc_pv,
                          (j > 0 || kk > 0) ? 1u : 0u);
              };
              tc_fence_after();
              if (elect_one()) issue_pv(0, kTileRows / 32);
              __syncwarp();
              if (!wait_warp(bar(C::kPFull + t), c[t] & 1, ctl, 0x207)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (elect_one()) {
                issue_pv(kTileRows / 32, kTileRows / 16);
                if (more) {
                  issue_s(t, qbase0, smem_u32(smem + C::kOffK + stn * C::kTileBytes));
                  umma_commit(bar(C::kSFull + t));
                } else {
                  umma_commit(bar(C::kOFull + t));
                }
                umma_commit(bar(C::kKVEmpty + st));   // this stage held sub-tile t's block only
              }
              __syncwarp();
              if (!more) ++e[t];
              ++c[t];
            }
          }
          if (!ok) break;
          if (elect_one()) umma_commit(bar(C::kQEmpty + qbuf));
          __syncwarp();
          g += ti.n0 + ti.n1;
          continue;
        }
        if (!wait_warp(bar(C::kKFull + g % C::kStages), (g / C::kStages) & 1, ctl, 0x202)) break;
        tc_fence_after();
        {
          const uint32_t kbase = smem_u32(smem + C::kOffK + (g % C::kStages) * C::kTileBytes);
          if (elect_one()) {
            for (int t = 0; t < 2; ++t) {
              if (n[t] == 0) continue;
              issue_s(t, qbase0 + t * C::kTileBytes, kbase);
              umma_commit(bar(C::kSFull + t));
            }
          }
          __syncwarp();
        }
        for (int j = 0; ok && j < ti.nkv; ++j) {
          const uint32_t gj = g + j;
          const int st = gj % C::kStages;
          const int stn = (gj + 1) % C::kStages;
          if (j + 1 < ti.nkv && !wait_warp(bar(C::kKFull + stn), ((gj + 1) / C::kStages) & 1, ctl, 0x203)) {
            ok = false;
            break;
          }
          if (!wait_warp(bar(C::kVFull + st), (gj / C::kStages) & 1, ctl, 0x204)) {
            ok = false;
            break;
          }
          const uint32_t vbase = smem_u32(smem + C::kOffV + st * C::kTileBytes);
          const uint32_t knext = smem_u32(smem + C::kOffK + stn * C::kTileBytes);
          // V's second 64-column block is the next 16 KB (d = 128) or the block of ones
          const uint32_t lbo = C::kOnesCol ? smem_u32(smem + C::kOffOnes) - vbase : kChunkBytes;
          const uint64_t vd = sdesc_sw128(vbase, lbo, 1024);
          // O_t += P_t V for keys [16*kk0, 16*kk1) of the block: B = V (keys x d), d
          // contiguous: MN-major; 16 keys = 16 rows of 128 bytes
          auto issue_pv = [&](int t, int kk0, int kk1) {
#pragma unroll
            for (int kk = kk0; kk < kk1; ++kk)
              umma_ts(tmem + C::tm_o(t), tmem + C::tm_p(t) + kk * 8, vd + ((kk * 16 * 128) >> 4), idesc_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
          };
          for (int t = 0; t < 2; ++t) {
            if (j >= n[t]) continue;
            // the first 64 keys' P are in tensor memory: their product overlaps the
            // softmax's exponentials of the other 64
            if (!wait_warp(bar(C::kPHalf + t), c[t] & 1, ctl, 0x205) ||
                (j == 0 && e[t] > 0 && !wait_warp(bar(C::kOEmpty + t), (e[t] - 1) & 1, ctl, 0x206))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) issue_pv(t, 0, kTileRows / 32);
            __syncwarp();
            if (!wait_warp(bar(C::kPFull + t), c[t] & 1, ctl, 0x207)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (elect_one()) {
              issue_pv(t, kTileRows / 32, kTileRows / 16);
              if (j + 1 < n[t]) {
                issue_s(t, qbase0 + t * C::kTileBytes, knext);
                umma_commit(bar(C::kSFull + t));
              } else {
                umma_commit(bar(C::kOFull + t));
              }
            }
            __syncwarp();
            if (j + 1 >= n[t]) ++e[t];
            ++c[t];
          }
          if (ok && elect_one()) umma_commit(bar(C::kKVEmpty + st));
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) umma_commit(bar(C::kQEmpty + qbuf));
        __syncwarp();
        g += ti.nkv;
      }
      // no MMA may still be running on tensor memory when the CTA tears down
      if (elect_one()) umma_commit(bar(C::kDrain));
      __syncwarp();
      mbar_wait(bar(C::kDrain), 0, drain, 0x2f1);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<kSoftmaxRegs>();
    const int t = warp >> 2;                          // sub-tile of this warpgroup
    const int tid = threadIdx.x & 127;                // row inside the sub-tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::tm_s(t);
    const uint32_t p_addr = tmem + lane_base + C::tm_p(t);
    const uint32_t o_addr = tmem + lane_base + C::tm_o(t);
    const uint64_t c2 = f2_pack(scale_log2, scale_log2);
    uint32_t c = 0;   // steps of this sub-tile (S-full / P-full phases)
    uint32_t e = 0;   // epilogues of this sub-tile
    uint32_t mc = 0;  // split tiles merged (sub-tile 0) or published (sub-tile 1)
    float* merge_m = reinterpret_cast<float*>(smem + C::kOffMerge);
    float* merge_l = merge_m + kTileRows;
    for (int k = 0, tile = persistent_tile(0); tile < ntiles; tile = persistent_tile(++k)) {
      const TileInfo ti = decode_tile<MODE>(tile, BH, H, G, Nq, Nk, CAUSAL, pairing);
      const int n = t == 0 ? ti.n0 : ti.n1;
      const int qb = t == 0 ? ti.qb0 : ti.qb1;
      const int row = qb * kTileRows + tid;
      if (n == 0) {
        // no row of this block sees a key (causal, Nk < Nq): O = 0 and lse = -inf
        if (GEN && (t == 0 || ti.has1) && row < Nq) {
          uint8_t* orow = reinterpret_cast<uint8_t*>(out) + ((size_t)ti.bh * Nq + row) * (D * 2);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) st_global_v4(orow + i * 16, 0u, 0u, 0u, 0u);
          lse[(size_t)ti.bh * Nq + row] = -INFINITY;
        }
        continue;
      }
      // last key visible to this thread's row, and to the block's first row (the same
      // for the whole warpgroup: key blocks ending past it take the masked path)
      const int lim_row = CAUSAL ? min(Nk - 1, row + (Nk - Nq)) : (Nk - 1);
      const int lim_blk = CAUSAL ? min(Nk - 1, qb * kTileRows + (Nk - Nq)) : (Nk - 1);
      (void)lim_blk;
      float m = -INFINITY;
      float l = 0.f;    // running sum of P as computed: lse = m + log2(l)
      float lr = 0.f;   // running sum of P as rounded for the MMA: O = (sum P V) / lr
      bool ok = true;
      for (int j = 0; j < n; ++j, ++c) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + t), c & 1, ctl, 0x301))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, sr + q * 32);
        tmem_ld_wait();
        reg_fence<128>(sr);
        float* s = reinterpret_cast<float*>(sr);
        const int kb = key_block(ti, j) + ((kSplit && t == 1) ? ti.koff1 : 0);
        const int kbase = kb * kTileRows;
        if (GEN ? (kbase + kTileRows - 1 > lim_blk) : ((kbase + kTileRows > Nk) || (CAUSAL && kb == qb))) {
#pragma unroll
          for (int q = 0; q < 128; ++q)
            if (kbase + q > lim_row) s[q] = -INFINITY;
        }
        // row maximum: three-input max tree
        float m3[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m3[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
        for (int q = 24; q < 120; q += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) m3[i] = fmax3(m3[i], s[q + i], s[q + 8 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) m3[i] = fmaxf(m3[i], s[120 + i]);
        const float mx = fmax3(fmax3(m3[0], m3[1], m3[2]), fmax3(m3[3], m3[4], m3[5]), fmaxf(m3[6], m3[7]));
        const float mc = mx * scale_log2;
        const float m_new = (mc > m + kRescaleThreshold<DT>) ? mc : m;
        // (a row that has seen no key yet keeps m = -inf: its P are 0 and alpha 1)
        const float alpha = (GEN && m_new == m) ? 1.0f : ex2_approx(m - m_new);
        const float nm = (GEN && m_new == -INFINITY) ? 0.0f : -m_new;
        const uint64_t nm2 = f2_pack(nm, nm);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          // O holds every earlier P.V (committed before this S); bring it to the new
          // maximum before this block's first P.V adds to it
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t orr[32];
            tmem_ld32(o_addr + q * 32, orr);
            tmem_ld_wait();
            reg_fence<32>(orr);
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(o_addr + q * 32, orr);
          }
          if constexpr (C::kOnesCol) {   // the P-sum columns follow O
            uint32_t orr[16];
            tmem_ld16(o_addr + D, orr);
            tmem_ld_wait();
            reg_fence<16>(orr);
#pragma unroll
            for (int i = 0; i < 16; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st16(o_addr + D, orr);
          }
        }
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};    // sum of P as computed (for lse)
        uint64_t accr[4] = {0ull, 0ull, 0ull, 0ull};   // d = 128: sum of P as rounded for the MMA
        // P in two halves of 64 keys; each half is handed to the MMA warp as soon as it
        // is in tensor memory
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int qq = hf * 32 + q;
            float x0, x1;
            f2_unpack(ffma2(f2_pack(s[2 * qq], s[2 * qq + 1]), c2, nm2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            acc[q & 3] = fadd2(acc[q & 3], f2_pack(p0, p1));
            pk[q] = pack2<DT>(p0, p1);
            if constexpr (!C::kOnesCol) accr[q & 3] = fadd2(accr[q & 3], unpack2_f2<DT>(pk[q]));
          }
          tmem_st32(p_addr + hf * 32, pk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(hf == 0 ? C::kPHalf + t : C::kPFull + t));
        }
        float a0, a1, b0, b1;
        f2_unpack(fadd2(acc[0], acc[1]), a0, a1);
        f2_unpack(fadd2(acc[2], acc[3]), b0, b1);
        const float rowsum = (a0 + a1) + (b0 + b1);
        l = l * alpha + rowsum;
        if constexpr (!C::kOnesCol) {
          f2_unpack(fadd2(accr[0], accr[1]), a0, a1);
          f2_unpack(fadd2(accr[2], accr[3]), b0, b1);
          lr = lr * alpha + ((a0 + a1) + (b0 + b1));
        }
        m = m_new;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kOFull + t), e & 1, ctl, 0x303))) break;
      ++e;
      tc_fence_after();
      if constexpr (kSplit) {
        if (t == 1) {
          // split tile: hand this half's running maximum and sum to sub-tile 0, which
          // merges the two halves (it reads O_1 from tensor memory: the same rows) and
          // frees both O buffers
          if (!__all_sync(0xffffffffu, mc == 0 || mbar_wait(bar(C::kMergeFree), (mc - 1) & 1, ctl, 0x305))) break;
          merge_m[tid] = m;
          merge_l[tid] = l;
          ++mc;
          mbar_arrive(bar(C::kMerge));
          continue;
        }
      }
      if constexpr (C::kOnesCol) {   // the MMA summed the 16-bit P values into O column D
        uint32_t orr[16];
        tmem_ld16(o_addr + D, orr);
        tmem_ld_wait();
        reg_fence<16>(orr);
        lr = __uint_as_float(orr[0]);
      }
      // split tile: m = max(m_0, m_1), O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (lr_0 2^(m_0 - m)
      // + lr_1 2^(m_1 - m)) and l likewise: the merge of two blocks' statistics
      const bool merge = kSplit && ti.n1 > 0;
      const uint32_t o1_addr = tmem + lane_base + C::tm_o(1);
      float a0 = 1.0f, a1 = 0.0f;
      if (merge) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kMerge), mc & 1, ctl, 0x306))) break;
        tc_fence_after();   // O_1 is complete: sub-tile 1 saw its last P.V before publishing
        ++mc;
        const float m1 = merge_m[tid], l1 = merge_l[tid];
        mbar_arrive(bar(C::kMergeFree));
        uint32_t orr[16];
        tmem_ld16(o1_addr + D, orr);   // sub-tile 1's sum of the 16-bit P values
        tmem_ld_wait();
        reg_fence<16>(orr);
        const float lr1 = __uint_as_float(orr[0]);
        const float mm = fmaxf(m, m1);
        a0 = m == -INFINITY ? 0.0f : ex2_approx(m - mm);
        a1 = m1 == -INFINITY ? 0.0f : ex2_approx(m1 - mm);
        l = l * a0 + l1 * a1;
        lr = lr * a0 + lr1 * a1;
        m = mm;
      }
      const float inv_l = (!GEN || lr > 0.0f) ? 1.0f / lr : 0.0f;   // a row that saw no key: O = 0
      uint8_t* orow = reinterpret_cast<uint8_t*>(out) + ((size_t)ti.bh * Nq + row) * (D * 2);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t orr[32];
        tmem_ld32(o_addr + q * 32, orr);
        tmem_ld_wait();
        reg_fence<32>(orr);
        if (merge) {
          uint32_t o1[32];
          tmem_ld32(o1_addr + q * 32, o1);
          tmem_ld_wait();
          reg_fence<32>(o1);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            orr[i] = __float_as_uint(fmaf(__uint_as_float(orr[i]), a0, __uint_as_float(o1[i]) * a1));
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<DT>(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
        if (row < Nq) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_global_v4(orow + q * 64 + i * 16, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row < Nq) lse[(size_t)ti.bh * Nq + row] = (m + lg2_approx(l)) * 0.69314718055994530942f;
      tc_fence_before();
      mbar_arrive(bar(C::kOEmpty + t));
      if (merge) mbar_arrive(bar(C::kOEmpty + 1));
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int DT, bool CAUSAL, int MODE, bool SPLIT>
cudaError_t launch_fwd_k(const FwdArgs& a, cudaStream_t stream, int pairing, int grid) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, DT, CAUSAL, MODE, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel must fit what the launch provides, or the
  // softmax warpgroups' setmaxnreg.inc would never be granted.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kThreads < (2 * kSoftmaxRegs + kOtherRegs) * 128) return cudaErrorInvalidConfiguration;
  return launch_overlapped(kern, grid, kThreads, C::kSmemBytes, stream, a.tm_q, a.tm_k, a.tm_v,
                           static_cast<uint16_t*>(a.o), a.lse, a.BH, a.H, a.G, a.Nq, a.Nk, a.scale_log2, pairing,
                           a.err_word, a.limit_ns);
}

template <int D, int DT, bool CAUSAL, int MODE>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  // (the butterfly pattern is defined on adjacent pairs of query blocks)
  int grid = 0;
  const int pairing = choose_pairing(a.BH, a.Nq, a.Nk, CAUSAL, MODE != 2, MODE != 2, a.num_sms, &grid);
  // single-block tiles at d = 64: the instance that splits each tile's key blocks between
  // the two sub-tiles (pairing 3), so that both softmax warpgroups work
  if constexpr (D == 64 && MODE != 2) {
    if (pairing == 2) return launch_fwd_k<D, DT, CAUSAL, MODE, true>(a, stream, 3, grid);
  }
  return launch_fwd_k<D, DT, CAUSAL, MODE, false>(a, stream, pairing, grid);
}

template <int MODE>
cudaError_t launch_fwd_g(const FwdArgs& a, cudaStream_t stream) {
  const int key = (a.d == 128 ? 4 : 0) | (a.dtype == 1 ? 2 : 0) | (a.causal ? 1 : 0);
  switch (key) {
    case 0: return launch_fwd_t<64, 0, false, MODE>(a, stream);
    case 1: return launch_fwd_t<64, 0, true, MODE>(a, stream);
    case 2: return launch_fwd_t<64, 1, false, MODE>(a, stream);
    case 3: return launch_fwd_t<64, 1, true, MODE>(a, stream);
    case 4: return launch_fwd_t<128, 0, false, MODE>(a, stream);
    case 5: return launch_fwd_t<128, 0, true, MODE>(a, stream);
    case 6: return launch_fwd_t<128, 1, false, MODE>(a, stream);
    default: return launch_fwd_t<128, 1, true, MODE>(a, stream);
  }
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.pattern == 1) return launch_fwd_g<2>(a, stream);
  return (a.Nq != a.Nk || a.G != 1) ? launch_fwd_g<1>(a, stream) : launch_fwd_g<0>(a, stream);
}

}  // namespace fa
