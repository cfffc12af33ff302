// fwd.cu -- forward kernel of exact tiled attention for sm_103a.
//
// One persistent CTA per SM walks (batch*head, 128-row query block) tiles, heaviest
// causal tiles first.  Inside a CTA the work is split by role:
//
//   warp 4      TMA producer: Q tile (double-buffered) and a ring of K/V stages.
//   warp 5      MMA issuer (one thread): S = Q K^T into tensor memory (double-
//               buffered), then O += P V with P read from tensor memory.
//   warps 0-3   softmax warpgroup, one thread per query row: reads its row of S
//               from tensor memory, applies the causal/tail mask, updates the
//               running maximum m and running sum l, writes P (16-bit) back to
//               tensor memory, rescales the unnormalised O when m moved, and in
//               the epilogue divides O by l and writes O and lse.
//
// The method follows the "Flash Attention" chapter (mlx.void.app): section
// "地基：流式 softmax" for the running (m, l) with the e^{m_old-m_new} patch,
// "FlashAttention——把整件事分块塞进 SRAM" for the query-outer / key-value-inner tiling
// in which the score tile never leaves the chip, and "FlashAttention-2" for the
// deferred division by l and the skipping of tiles wholly above the causal
// diagonal.  Exponentials are taken in base 2 with scale*log2(e) folded into one
// FMA (2^{x log2 e} = e^x).
//
// The running maximum is only moved when a new row maximum exceeds it by more than
// 8 (base-2 units).  Until then P entries may reach 2^8; the result is unchanged
// because l and O are accumulated against the same maximum, and O's rescale in
// tensor memory is skipped on most blocks.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kTileRows = 128;   // query rows per tile and keys per key/value block
constexpr int kThreads = 192;    // 4 softmax warps + producer warp + MMA warp
constexpr int kChunkBytes = kTileRows * 128;   // one 128-row x 128-byte swizzle column block
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;                    // 64 16-bit elements per 128-byte row
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;                          // [2]
  static constexpr int kQEmpty = 2;                         // [2]
  static constexpr int kKFull = 4;                          // [kStages]
  static constexpr int kVFull = kKFull + kStages;           // [kStages]
  static constexpr int kKVEmpty = kVFull + kStages;         // [kStages]
  static constexpr int kSFull = kKVEmpty + kStages;         // [2]
  static constexpr int kPFull = kSFull + 2;                 // [2]
  static constexpr int kPVDone = kPFull + 2;
  static constexpr int kOEmpty = kPVDone + 1;
  static constexpr int kDrain = kOEmpty + 1;
  static constexpr int kNumBars = kDrain + 1;
  // + alignment slack; d = 64 also keeps 32 KB after the last V stage so that every
  // operand read an MMA descriptor can address stays inside this CTA's allocation
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024 + (D == 64 ? 32768 : 0);
  // tensor memory columns (512 allocated)
  static constexpr uint32_t kTmS = 0;      // S buffers at 0 and 128 (fp32)
  static constexpr uint32_t kTmP = 256;    // P buffers at 256 and 320 (16-bit pairs)
  static constexpr uint32_t kTmO = 384;    // O accumulator, D columns (fp32)
};

__device__ __forceinline__ void decode_tile(int tile, int BH, int nqb, int& bh, int& qb) {
  const int r = tile / BH;   // r = 0 holds the last (heaviest, causal) query block of every head
  bh = tile - r * BH;
  qb = nqb - 1 - r;
}

template <int D, int DT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, uint16_t* __restrict__ out, float* __restrict__ lse,
               int BH, int N, float scale_log2, unsigned int* err_word, uint64_t limit_ns) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqb = (N + kTileRows - 1) / kTileRows;
  const int ntiles = BH * nqb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kQFull + i), 1);
      mbar_init(bar(C::kQEmpty + i), 1);
      mbar_init(bar(C::kSFull + i), 1);
      mbar_init(bar(C::kPFull + i), kTileRows);
    }
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bar(C::kKFull + i), 1);
      mbar_init(bar(C::kVFull + i), 1);
      mbar_init(bar(C::kKVEmpty + i), 1);
    }
    mbar_init(bar(C::kPVDone), 1);
    mbar_init(bar(C::kOEmpty), kTileRows);
    mbar_init(bar(C::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl ctl{abort_flag, err_word, limit_ns};
  const WaitCtl drain{nullptr, err_word, limit_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++it) {
        int bh, qb;
        decode_tile(tile, BH, nqb, bh, qb);
        const int nkv = CAUSAL ? qb + 1 : nqb;
        const int qbuf = it & 1;
        if (it >= 2 && !mbar_wait(bar(C::kQEmpty + qbuf), ((it >> 1) - 1) & 1, ctl, 0x101)) {
          ok = false;
          break;
        }
        const uint32_t qdst = smem_u32(smem + C::kOffQ + qbuf * C::kTileBytes);
        mbar_arrive_expect_tx(bar(C::kQFull + qbuf), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(qdst + c * kChunkBytes, &tm_q, bar(C::kQFull + qbuf), c * 64, qb * kTileRows, bh);
        for (int j = 0; j < nkv; ++j, ++g) {
          const int st = g % C::kStages;
          if (g >= (uint32_t)C::kStages &&
              !mbar_wait(bar(C::kKVEmpty + st), ((g / C::kStages) - 1) & 1, ctl, 0x102)) {
            ok = false;
            break;
          }
          const uint32_t kdst = smem_u32(smem + C::kOffK + st * C::kTileBytes);
          const uint32_t vdst = smem_u32(smem + C::kOffV + st * C::kTileBytes);
          mbar_arrive_expect_tx(bar(C::kKFull + st), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(kdst + c * kChunkBytes, &tm_k, bar(C::kKFull + st), c * 64, j * kTileRows, bh);
          mbar_arrive_expect_tx(bar(C::kVFull + st), C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(vdst + c * kChunkBytes, &tm_v, bar(C::kVFull + st), c * 64, j * kTileRows, bh);
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
        for (int qb2 = 0; qb2 < 2; ++qb2) {
          if (it > qb2) {
            const int last = it - 1 - ((it - 1 - qb2) & 1);
            mbar_wait(bar(C::kQFull + qb2), (last >> 1) & 1, drain, 0x1f3);
          }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ab = (DT == 0) ? 1u : 0u;   // instruction-descriptor code: bf16 = 1, fp16 = 0
      constexpr uint32_t idesc_qk = idesc_f16(ab, 0, 0, 128, 128);
      constexpr uint32_t idesc_pv = idesc_f16(ab, 0, 1, 128, D);
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t gp, int jp) -> bool {
        const int sb = gp & 1;
        const int st = gp % C::kStages;
        if (!mbar_wait(bar(C::kPFull + sb), (gp >> 1) & 1, ctl, 0x201)) return false;
        if (!mbar_wait(bar(C::kVFull + st), (gp / C::kStages) & 1, ctl, 0x202)) return false;
        if (jp == 0 && it > 0 && !mbar_wait(bar(C::kOEmpty), (it - 1) & 1, ctl, 0x203)) return false;
        tc_fence_after();
        const uint32_t vbase = smem_u32(smem + C::kOffV + st * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk) {
          // B = V (keys x d), d contiguous: MN-major; 16 keys = 16 rows of 128 bytes
          const uint64_t bdesc = sdesc_sw128(vbase + kk * 16 * 128, kChunkBytes, 1024);
          umma_ts(tmem + C::kTmO, tmem + C::kTmP + sb * 64 + kk * 8, bdesc, idesc_pv,
                  (jp > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(C::kPVDone));
        umma_commit(bar(C::kKVEmpty + st));
        return true;
      };
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++it) {
        int bh, qb;
        decode_tile(tile, BH, nqb, bh, qb);
        const int nkv = CAUSAL ? qb + 1 : nqb;
        const int qbuf = it & 1;
        if (!mbar_wait(bar(C::kQFull + qbuf), (it >> 1) & 1, ctl, 0x204)) break;
        const uint32_t qbase = smem_u32(smem + C::kOffQ + qbuf * C::kTileBytes);
        for (int j = 0; j < nkv; ++j, ++g) {
          const int st = g % C::kStages;
          if (!mbar_wait(bar(C::kKFull + st), (g / C::kStages) & 1, ctl, 0x205)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + C::kOffK + st * C::kTileBytes);
          const uint32_t d_s = tmem + C::kTmS + (g & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // A = Q (rows x d), B = K (keys x d): both K-major; 16 elements = 32 bytes
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            umma_ss(d_s, sdesc_sw128(qbase + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_qk,
                    kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(C::kSFull + (g & 1)));
          if (j == nkv - 1) umma_commit(bar(C::kQEmpty + qbuf));
          if (j > 0 && !issue_pv(g - 1, j - 1)) {
            ok = false;
            break;
          }
        }
        if (ok && !issue_pv(g - 1, nkv - 1)) ok = false;
      }
      // no MMA may still be running on tensor memory when the CTA tears down
      umma_commit(bar(C::kDrain));
      mbar_wait(bar(C::kDrain), 0, drain, 0x2f1);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int t = threadIdx.x;                       // row inside the tile
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t g = 0;
    uint32_t pv_phase = 0;                           // completed PV-done phases waited so far
    int it = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
      int bh, qb;
      decode_tile(tile, BH, nqb, bh, qb);
      const int nkv = CAUSAL ? qb + 1 : nqb;
      const int row = qb * kTileRows + t;
      float m = -INFINITY;
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv; ++j, ++g) {
        const int sb = g & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + sb), (g >> 1) & 1, ctl, 0x301))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + C::kTmS + sb * 128 + c * 32, sr + c * 32);
        tmem_ld_wait();
        reg_fence<128>(sr);
        float* s = reinterpret_cast<float*>(sr);
        const int kbase = j * kTileRows;
        const bool tail = (kbase + kTileRows > N);
        const bool diag = CAUSAL && (j == qb);
        if (tail || diag) {
          const int lim = CAUSAL ? min(N - 1, row) : (N - 1);   // last visible key
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (kbase + c > lim) s[c] = -INFINITY;
        }
        // row maximum: 8 independent chains, then a tree
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int c = 8; c < 128; c += 8)
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[c + i]);
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float mc = mx * scale_log2;
        const float m_new = (mc > m + kRescaleThreshold) ? mc : m;
        const float alpha = ex2_approx(m - m_new);
        const float neg_m = -m_new;
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2_approx(fmaf(s[2 * c], scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(s[2 * c + 1], scale_log2, neg_m));
          l8[(2 * c) & 7] += p0;
          l8[(2 * c + 1) & 7] += p1;
          pk[c] = pack2<DT>(p0, p1);
        }
        const float rowsum = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        l = l * alpha + rowsum;
        tmem_st32(tmem + lane_base + C::kTmP + sb * 64, pk);
        tmem_st32(tmem + lane_base + C::kTmP + sb * 64 + 32, pk + 32);
        if (j > 0) {
          // the previous P.V must have landed in O before O is rescaled
          if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kPVDone), pv_phase & 1, ctl, 0x302))) {
            ok = false;
            break;
          }
          ++pv_phase;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(tmem + lane_base + C::kTmO + c * 32, orr);
              tmem_ld_wait();
              reg_fence<32>(orr);
#pragma unroll
              for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
              tmem_st32(tmem + lane_base + C::kTmO + c * 32, orr);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kPFull + sb));
        m = m_new;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kPVDone), pv_phase & 1, ctl, 0x303))) break;
      ++pv_phase;
      tc_fence_after();
      const float inv_l = 1.0f / l;
      uint8_t* orow = reinterpret_cast<uint8_t*>(out) + ((size_t)bh * N + row) * (D * 2);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(tmem + lane_base + C::kTmO + c * 32, orr);
        tmem_ld_wait();
        reg_fence<32>(orr);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<DT>(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
        if (row < N) {
#pragma unroll
          for (int i = 0; i < 4; ++i) st_global_v4(orow + c * 64 + i * 16, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row < N) lse[(size_t)bh * N + row] = (m + lg2_approx(l)) * 0.69314718055994530942f;
      tc_fence_before();
      mbar_arrive(bar(C::kOEmpty));
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int DT, bool CAUSAL>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, DT, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nqb = (a.N + kTileRows - 1) / kTileRows;
  const int ntiles = a.BH * nqb;
  const int grid = ntiles < a.num_sms ? ntiles : a.num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(a.tm_q, a.tm_k, a.tm_v, static_cast<uint16_t*>(a.o), a.lse,
                                                   a.BH, a.N, a.scale_log2, a.err_word, a.limit_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  const int key = (a.d == 128 ? 4 : 0) | (a.dtype == 1 ? 2 : 0) | (a.causal ? 1 : 0);
  switch (key) {
    case 0: return launch_fwd_t<64, 0, false>(a, stream);
    case 1: return launch_fwd_t<64, 0, true>(a, stream);
    case 2: return launch_fwd_t<64, 1, false>(a, stream);
    case 3: return launch_fwd_t<64, 1, true>(a, stream);
    case 4: return launch_fwd_t<128, 0, false>(a, stream);
    case 5: return launch_fwd_t<128, 0, true>(a, stream);
    case 6: return launch_fwd_t<128, 1, false>(a, stream);
    default: return launch_fwd_t<128, 1, true>(a, stream);
  }
}

}  // namespace fa
