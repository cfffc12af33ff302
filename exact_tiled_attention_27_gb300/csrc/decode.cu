// decode.cu -- split-key attention for a few query rows (decoding) on sm_103a.
//
// When each key/value head has only a handful of query rows (G = H/Hkv query heads
// of a group times Nq new tokens, at most 8 rows), attention is a pass over K and V
// that touches every element once: it is bound by device-memory bandwidth, not by
// arithmetic, so it runs on the CUDA cores instead of padding the rows out to a 128-row
// tensor-core tile.  To occupy every SM even for a few heads, the keys of a head are
// cut into S contiguous ranges ("splits"), one CTA per (split, key/value head):
//
//   decode_split_kernel   for its key range: the scores, the streaming (m, l)
//                         softmax and the unnormalised sum of P V for each query row,
//                         then O_s = sum / l and lse_s = m + ln l of that range.
//   decode_merge_kernel   (S > 1) combines the ranges: lse = ln sum_s e^{lse_s},
//                         O = sum_s e^{lse_s - lse} O_s -- the merge of two blocks'
//                         statistics in the FlashAttention review ("方法细节"), applied
//                         to whole key ranges.
//
// The streaming update is the one of the "Flash Attention" chapter ("地基：流式
// softmax"), taken 32 keys at a time per row and in base 2 (scale*log2(e) is folded
// into Q); the running maximum only moves when a score exceeds it by more than 8.  The
// causal mask is aligned bottom-right (query i of Nq sees key j iff j <= i + Nk - Nq),
// so a single new token sees the whole cache.
//
// Inside a range a producer warp streams the keys in stages of 32 rows (K and V, 64-column
// blocks with the 128-byte swizzle) through a ring of shared-memory stages with the tensor
// memory accelerator, and kDecWarps consumer warps take the stages in turn (stage s to warp
// s mod kDecWarps).  The bytes in flight sit in shared memory, not registers, so one CTA
// per SM keeps the device memory busy.  On its stage a consumer warp computes the scores
// with one key per lane (its K row, read conflict-free from the swizzled layout, against the
// query rows broadcast from shared memory), so a score needs no cross-lane sum; the running
// maximum moves once per 32 keys (one warp reduction per query row); for P V each lane owns
// D/32 columns of every query row and reads those columns of the 32 V rows and the 32
// probabilities from shared memory.  The products use the paired float32 FMA (two columns
// per instruction).  Each warp keeps its own (m, l, O) over the keys it visited; the CTA
// merges its warps at the end.
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kDecThreshold = 8.0f;
constexpr float kDecLn2 = 0.69314718055994530942f;
constexpr float kDecLog2e = 1.4426950408889634f;

// Query row m of key/value head bhk = b * Hkv + hk: query head hk*G + m/Nq, position m%Nq.
__device__ __forceinline__ size_t query_row(int bhk, int m, int H, int Hkv, int Nq) {
  const int b = bhk / Hkv, hk = bhk - b * Hkv, G = H / Hkv;
  const int g = m / Nq, qi = m - g * Nq;
  return (size_t)(b * H + hk * G + g) * Nq + qi;
}

// Every ring slot belongs to one consumer warp, so a warp waits on a slot only after it
// has itself consumed the slot's previous use: a parity wait can then never be satisfied
// by a phase that is one use behind.  Twelve warps with one slot each (16 KB at d = 128)
// keep three consumer warps on every scheduler while eleven slots are in flight.  (Six
// warps with two slots each: -1 % with 4 query rows and -9 % with 8, where the warps'
// arithmetic is the longer part.)
constexpr int kDecWarps = 12;
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecSlotsPerWarp = 1;
constexpr int kDecStages = kDecSlotsPerWarp * kDecWarps;
// ring slot of stage s (its consuming warp's slot for that warp's (s / kDecWarps)-th
// stage) and the use of that slot it is
__device__ __forceinline__ int dec_slot(int s) {
  return (s % kDecWarps) + kDecWarps * ((s / kDecWarps) % kDecSlotsPerWarp);
}
__device__ __forceinline__ int dec_use(int s) { return (s / kDecWarps) / kDecSlotsPerWarp; }

template <int D>
struct DecCfg {
  static constexpr int kBlock = 32 * 128;             // 32 rows x one 64-column block (128 bytes)
  static constexpr int kHalf = (D / 64) * kBlock;     // K, or V, of one stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kOffBar = kDecStages * kStage;
  static constexpr int kSmem = kOffBar + 2 * kDecStages * 8 + 1024;   // + alignment slack
};

template <int D, int DT, int MR>
__global__ void __launch_bounds__(kDecThreads, 1) decode_split_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, float* __restrict__ opart, float* __restrict__ lpart,
    uint16_t* __restrict__ out, float* __restrict__ lse, int H, int Hkv, int Nq, int Nk, int M, int chunk,
    float scale_log2, int causal, unsigned int* err_word, uint64_t limit_ns) {
  using C = DecCfg<D>;
  constexpr int kCols = D / 32;                // output columns per lane
  __shared__ __align__(16) float sq[MR][D];    // query rows times scale*log2(e)
  __shared__ __align__(16) float sp[kDecWarps][32][MR];
  __shared__ float sm_m[kDecWarps][MR];
  __shared__ float sm_l[kDecWarps][MR];
  __shared__ int abort_flag;
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* ring = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::kOffBar);
  auto full = [&](int i) { return smem_u32(bars + i); };
  auto empty = [&](int i) { return smem_u32(bars + kDecStages + i); };

  const int split = blockIdx.x, S = gridDim.x;
  const int bhk = blockIdx.y, BHkv = gridDim.y;
  const int lane = threadIdx.x & 31;
  const int warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const int k0 = split * chunk;
  const int k1 = min(Nk, k0 + chunk);
  const int nst = (k1 - k0 + 31) / 32;         // stages of this range
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  grid_dep_wait();
  for (int i = threadIdx.x; i < MR * (D / 8); i += kDecThreads) {
    const int m = i / (D / 8), c8 = i % (D / 8);
    float f8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (m < M) {
      const uint4 w = *reinterpret_cast<const uint4*>(q + query_row(bhk, m, H, Hkv, Nq) * D + c8 * 8);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = unpack2<DT>(ww[c]);
        f8[2 * c] = f.x * scale_log2;
        f8[2 * c + 1] = f.y * scale_log2;
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) sq[m][c8 * 8 + c] = f8[c];
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, err_word, limit_ns};
  const WaitCtl drain{nullptr, err_word, limit_ns};

  float mrow[MR], lrow[MR];
  uint64_t acc2[MR][kCols / 2];   // this lane's columns of O, in pairs
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    mrow[m] = -INFINITY;
    lrow[m] = 0.f;   // this lane's share of l
#pragma unroll
    for (int c = 0; c < kCols / 2; ++c) acc2[m][c] = 0ull;
  }

  if (warp == kDecWarps) {
    // ---------------------------------------------------------- producer (one lane issues)
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    bool ok = true;
    int s = 0;
    for (; s < nst; ++s) {
      const int slot = dec_slot(s);
      if (s >= kDecStages && !wait_warp(empty(slot), (dec_use(s) - 1) & 1, ctl, 0x801)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t dst = smem_u32(ring + slot * C::kStage);
        mbar_arrive_expect_tx(full(slot), C::kStage);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(dst + c * C::kBlock, &tm_k, full(slot), c * 64, k0 + 32 * s, bhk);
          tma_load_3d(dst + C::kHalf + c * C::kBlock, &tm_v, full(slot), c * 64, k0 + 32 * s, bhk);
        }
      }
      __syncwarp();
    }
    if (!ok) {   // every copy already issued must land before the ring is reused below
      for (int t = (s > kDecStages ? s - kDecStages : 0); t < s; ++t)
        mbar_wait(full(dec_slot(t)), dec_use(t) & 1, drain, 0x8f1);
    }
  } else {
    // ---------------------------------------------------------- consumers
    int lim[MR];   // last key each query row sees (-1: a padding row sees none)
#pragma unroll
    for (int m = 0; m < MR; ++m) lim[m] = m < M ? (causal ? (m % Nq) + (Nk - Nq) : Nk - 1) : -1;
    float* pw = &sp[warp][0][0];
    for (int s = warp; s < nst; s += kDecWarps) {
      const int slot = dec_slot(s);
      if (!wait_warp(full(slot), dec_use(s) & 1, ctl, 0x802)) break;
      const uint8_t* kbuf = ring + slot * C::kStage;
      const uint8_t* vbuf = kbuf + C::kHalf;
      const int j0 = k0 + 32 * s;
      const int j = j0 + lane;
      const bool live = j < k1;
      uint64_t dot2[MR];   // (even columns, odd columns) partial dot products
#pragma unroll
      for (int m = 0; m < MR; ++m) dot2[m] = 0ull;
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) {
        // this lane's key row, 16 bytes of it: block c8/8, swizzled unit (c8 % 8) ^ (row % 8)
        const uint4 kr = *reinterpret_cast<const uint4*>(kbuf + (c8 >> 3) * C::kBlock + lane * 128 +
                                                         (((c8 & 7) ^ (lane & 7)) << 4));
        const uint64_t k2[4] = {unpack2_f2<DT>(kr.x), unpack2_f2<DT>(kr.y), unpack2_f2<DT>(kr.z),
                                unpack2_f2<DT>(kr.w)};
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(&sq[m][c8 * 8]);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(&sq[m][c8 * 8 + 4]);
          dot2[m] = ffma2(qa.x, k2[0], dot2[m]);
          dot2[m] = ffma2(qa.y, k2[1], dot2[m]);
          dot2[m] = ffma2(qb.x, k2[2], dot2[m]);
          dot2[m] = ffma2(qb.y, k2[3], dot2[m]);
        }
      }
      float dot[MR];
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        float lo, hi;
        f2_unpack(dot2[m], lo, hi);
        dot[m] = lo + hi;
      }
      // ---- streaming softmax over the 32 keys (the maximum moves at most once per row)
      float p[MR];
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float x = (live && j <= lim[m]) ? dot[m] : -INFINITY;
        float bm = x;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        if (bm > mrow[m] + kDecThreshold) {   // e^{m_old - m_new} patch of l and O
          const float a = ex2_approx(mrow[m] - bm);
          lrow[m] *= a;
          const uint64_t a2 = f2_pack(a, a);
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) acc2[m][c] = fmul2(acc2[m][c], a2);
          mrow[m] = bm;
        }
        p[m] = x == -INFINITY ? 0.f : ex2_approx(x - mrow[m]);
        lrow[m] += p[m];
      }
      if constexpr (MR >= 4) {
#pragma unroll
        for (int m4 = 0; m4 < MR; m4 += 4)
          *reinterpret_cast<float4*>(pw + lane * MR + m4) = make_float4(p[m4], p[m4 + 1], p[m4 + 2], p[m4 + 3]);
      } else {
#pragma unroll
        for (int m = 0; m < MR; ++m) pw[lane * MR + m] = p[m];
      }
      __syncwarp();
      // ---- O += P V: this lane's columns of the 32 V rows (rows past the range have P = 0)
      const int vcol = lane * kCols;
      const int vblk = vcol >> 6, vbyte = (vcol & 63) * 2;
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const uint8_t* vrow = vbuf + vblk * C::kBlock + kk * 128 + ((((vbyte >> 4) ^ (kk & 7)) << 4) | (vbyte & 15));
        uint64_t v2[kCols / 2];
        if constexpr (kCols == 2) {
          v2[0] = unpack2_f2<DT>(*reinterpret_cast<const uint32_t*>(vrow));
        } else {
          const uint2 w2 = *reinterpret_cast<const uint2*>(vrow);
          v2[0] = unpack2_f2<DT>(w2.x);
          v2[1] = unpack2_f2<DT>(w2.y);
        }
        float pk[MR];
        if constexpr (MR >= 4) {
#pragma unroll
          for (int m4 = 0; m4 < MR; m4 += 4) {
            const float4 x = *reinterpret_cast<const float4*>(pw + kk * MR + m4);
            pk[m4] = x.x;
            pk[m4 + 1] = x.y;
            pk[m4 + 2] = x.z;
            pk[m4 + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int m = 0; m < MR; ++m) pk[m] = pw[kk * MR + m];
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const uint64_t p2 = f2_pack(pk[m], pk[m]);
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) acc2[m][c] = ffma2(p2, v2[c], acc2[m][c]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(slot));
    }
  }
  // every stage has been read (or the ring drained): its memory now holds the warps' sums
  __syncthreads();
  float* sm_acc = reinterpret_cast<float*>(ring);   // [kDecWarps][MR][D]
  if (warp < kDecWarps) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lrow[m] += __shfl_xor_sync(0xffffffffu, lrow[m], off);
#pragma unroll
      for (int c = 0; c < kCols / 2; ++c) {
        float lo, hi;
        f2_unpack(acc2[m][c], lo, hi);
        sm_acc[(warp * MR + m) * D + lane * kCols + 2 * c] = lo;
        sm_acc[(warp * MR + m) * D + lane * kCols + 2 * c + 1] = hi;
      }
      if (lane == 0) {
        sm_m[warp][m] = mrow[m];
        sm_l[warp][m] = lrow[m];
      }
    }
  }
  __syncthreads();
  // merge the warps: one thread per (query row, 8 columns)
  if (threadIdx.x < M * (D / 8)) {
    const int m = threadIdx.x / (D / 8), rr = threadIdx.x % (D / 8);
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, sm_m[w][m]);
    float lsum = 0.f, a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float sc = sm_m[w][m] == -INFINITY ? 0.f : ex2_approx(sm_m[w][m] - mx);
      lsum += sm_l[w][m] * sc;
#pragma unroll
      for (int c = 0; c < 8; ++c) a[c] += sm_acc[(w * MR + m) * D + rr * 8 + c] * sc;
    }
    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;                    // no visible key: O = 0
    const float lse_v = lsum > 0.f ? (mx + lg2_approx(lsum)) * kDecLn2 : -INFINITY;
    if (S == 1) {
      const size_t row = query_row(bhk, m, H, Hkv, Nq);
      uint4 w;
      w.x = pack2<DT>(a[0] * inv, a[1] * inv);
      w.y = pack2<DT>(a[2] * inv, a[3] * inv);
      w.z = pack2<DT>(a[4] * inv, a[5] * inv);
      w.w = pack2<DT>(a[6] * inv, a[7] * inv);
      *reinterpret_cast<uint4*>(out + row * D + rr * 8) = w;
      if (rr == 0) lse[row] = lse_v;
    } else {
      const size_t prow = ((size_t)split * BHkv + bhk) * M + m;
      float4* dst = reinterpret_cast<float4*>(opart + prow * D + rr * 8);
      dst[0] = make_float4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
      dst[1] = make_float4(a[4] * inv, a[5] * inv, a[6] * inv, a[7] * inv);
      if (rr == 0) lpart[prow] = lse_v;
    }
  }
  grid_dep_launch();
}

// One thread per (key/value head, query row, 8-column segment): combine the S ranges.
template <int D, int DT>
__global__ void __launch_bounds__(256) decode_merge_kernel(const float* __restrict__ opart,
                                                           const float* __restrict__ lpart, uint16_t* __restrict__ out,
                                                           float* __restrict__ lse, int BHkv, int H, int Hkv, int Nq,
                                                           int M, int S) {
  constexpr int kTPK = D / 8;
  grid_dep_wait();
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  if (gtid < BHkv * M * kTPK) {
    const int rr = gtid % kTPK;
    const int prow = gtid / kTPK;             // bhk * M + m
    const int m = prow % M, bhk = prow / M;
    const size_t stride = (size_t)BHkv * M;
    float mx = -INFINITY;
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, lpart[s * stride + prow]);
    float wsum = 0.f, a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const float ls = lpart[s * stride + prow];
      const float w = ls == -INFINITY ? 0.f : ex2_approx((ls - mx) * kDecLog2e);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(opart + (s * stride + prow) * D + rr * 8);
      const float4 x0 = src[0], x1 = src[1];
      a[0] = fmaf(w, x0.x, a[0]);
      a[1] = fmaf(w, x0.y, a[1]);
      a[2] = fmaf(w, x0.z, a[2]);
      a[3] = fmaf(w, x0.w, a[3]);
      a[4] = fmaf(w, x1.x, a[4]);
      a[5] = fmaf(w, x1.y, a[5]);
      a[6] = fmaf(w, x1.z, a[6]);
      a[7] = fmaf(w, x1.w, a[7]);
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const size_t row = query_row(bhk, m, H, Hkv, Nq);
    uint4 w;
    w.x = pack2<DT>(a[0] * inv, a[1] * inv);
    w.y = pack2<DT>(a[2] * inv, a[3] * inv);
    w.z = pack2<DT>(a[4] * inv, a[5] * inv);
    w.w = pack2<DT>(a[6] * inv, a[7] * inv);
    *reinterpret_cast<uint4*>(out + row * D + rr * 8) = w;
    if (rr == 0) lse[row] = wsum > 0.f ? mx + lg2_approx(wsum) * kDecLn2 : -INFINITY;
  }
  grid_dep_launch();
}

template <int D, int DT, int MR>
cudaError_t launch_decode_t(const DecArgs& a, cudaStream_t stream) {
  auto kern = decode_split_kernel<D, DT, MR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(kern, dim3(a.S, a.BHkv), kDecThreads, DecCfg<D>::kSmem, stream, a.tm_k, a.tm_v,
                        static_cast<const uint16_t*>(a.q), a.opart, a.lpart, static_cast<uint16_t*>(a.o), a.lse, a.H,
                        a.Hkv, a.Nq, a.Nk, a.M, a.chunk, a.scale_log2, a.causal, a.err_word, a.limit_ns);
  if (e != cudaSuccess || a.S == 1) return e;
  const long long threads = (long long)a.BHkv * a.M * (D / 8);
  return launch_overlapped(decode_merge_kernel<D, DT>, dim3((unsigned)((threads + 255) / 256)), 256, 0, stream,
                           static_cast<const float*>(a.opart), static_cast<const float*>(a.lpart),
                           static_cast<uint16_t*>(a.o), a.lse, a.BHkv, a.H, a.Hkv, a.Nq, a.M, a.S);
}

template <int D, int DT>
cudaError_t launch_decode_m(const DecArgs& a, cudaStream_t stream) {
  if (a.M <= 1) return launch_decode_t<D, DT, 1>(a, stream);
  if (a.M <= 2) return launch_decode_t<D, DT, 2>(a, stream);
  if (a.M <= 4) return launch_decode_t<D, DT, 4>(a, stream);
  return launch_decode_t<D, DT, 8>(a, stream);
}

}  // namespace

cudaError_t launch_decode(const DecArgs& a, cudaStream_t stream) {
  const int key = (a.d == 128 ? 2 : 0) | (a.dtype == 1 ? 1 : 0);
  switch (key) {
    case 0: return launch_decode_m<64, 0>(a, stream);
    case 1: return launch_decode_m<64, 1>(a, stream);
    case 2: return launch_decode_m<128, 0>(a, stream);
    default: return launch_decode_m<128, 1>(a, stream);
  }
}

}  // namespace fa
