// decode.cu -- split-key attention for a few query rows (decoding) on sm_103a.
//
// When each key/value head has only a handful of query rows (G = H/Hkv query heads
// of a group times Nq new tokens, at most 8 rows), attention is a pass over K and V
// that touches every element once: it is bound by device-memory bandwidth, not by
// arithmetic, so it runs on the CUDA cores with coalesced 16-byte loads instead of
// padding the rows out to a 128-row tensor-core tile.  To occupy every SM even for a
// few heads, the keys of a head are cut into S contiguous ranges ("splits"), one CTA
// per (split, key/value head):
//
//   decode_split_kernel_* for its key range: the scores, the streaming (m, l)
//                         softmax and the unnormalised sum of P V for each query row,
//                         then O_s = sum / l and lse_s = m + ln l of that range.
//   decode_merge_kernel   (S > 1) combines the ranges: lse = ln sum_s e^{lse_s},
//                         O = sum_s e^{lse_s - lse} O_s -- the merge of two blocks'
//                         statistics in the FlashAttention review ("方法细节"), applied
//                         to whole key ranges.
//
// The streaming update is the one of the "Flash Attention" chapter ("地基：流式
// softmax"), taken one key at a time per row and in base 2 (scale*log2(e) is folded
// into Q); the running maximum only moves when a score exceeds it by more than 8, as
// in the forward kernel.  The causal mask is aligned bottom-right (query i of Nq sees
// key j iff j <= i + Nk - Nq), so a single new token sees the whole cache.
//
// Work split inside decode_split: a warp takes 32 consecutive keys at a time.
// For the scores each lane owns one key (its row of K is read 16 bytes at a time, the
// query rows are broadcast from shared memory), so a score needs no cross-lane sum;
// the running maximum moves once per 32 keys (one warp reduction per query row).  For
// P V each lane owns D/32 columns of every query row, reads those columns of the 32
// V rows (coalesced) and the 32 probabilities from shared memory.  Each warp keeps
// its own (m, l, O) over the keys it visited; the CTA merges its warps at the end.
#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr float kDecThreshold = 8.0f;
constexpr float kDecLn2 = 0.69314718055994530942f;
constexpr float kDecLog2e = 1.4426950408889634f;

// Query row m of key/value head bhk = b * Hkv + hk: query head hk*G + m/Nq, position m%Nq.
__device__ __forceinline__ size_t query_row(int bhk, int m, int H, int Hkv, int Nq) {
  const int b = bhk / Hkv, hk = bhk - b * Hkv, G = H / Hkv;
  const int g = m / Nq, qi = m - g * Nq;
  return (size_t)(b * H + hk * G + g) * Nq + qi;
}

// d = 64: each lane's V columns of the step are requested up front with its K row (32
// more registers; one CTA per SM keeps enough bytes in flight).  d = 128: that would cost
// 64 registers and the CTAs per SM that hide the latency, so V is read in the P V loop.
template <int D, int DT, int MR>
__device__ __forceinline__ void decode_split(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    float* __restrict__ opart, float* __restrict__ lpart, uint16_t* __restrict__ out, float* __restrict__ lse,
    int H, int Hkv, int Nq, int Nk, int M, int chunk, float scale_log2, int causal) {
  constexpr int kCols = D / 32;                // output columns per lane
  constexpr bool kVEarly = (D == 64);
  __shared__ __align__(16) float sq[MR][D];    // query rows times scale*log2(e)
  __shared__ __align__(16) float sp[kDecWarps][32][MR];
  __shared__ float sm_m[kDecWarps][MR];
  __shared__ float sm_l[kDecWarps][MR];
  __shared__ __align__(16) float sm_acc[kDecWarps][MR][D];

  grid_dep_wait();
  const int split = blockIdx.x, S = gridDim.x;
  const int bhk = blockIdx.y, BHkv = gridDim.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k0 = split * chunk;
  const int k1 = min(Nk, k0 + chunk);

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
  int lim[MR];   // last key each query row sees (-1: a padding row sees none)
#pragma unroll
  for (int m = 0; m < MR; ++m) lim[m] = m < M ? (causal ? (m % Nq) + (Nk - Nq) : Nk - 1) : -1;
  __syncthreads();

  float mrow[MR], lrow[MR], acc[MR][kCols];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    mrow[m] = -INFINITY;
    lrow[m] = 0.f;   // this lane's share of l
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[m][c] = 0.f;
  }
  const uint16_t* kh = k + (size_t)bhk * Nk * D;
  const uint16_t* vh = v + (size_t)bhk * Nk * D;
  float* pw = &sp[warp][0][0];

  for (int j0 = k0 + warp * 32; j0 < k1; j0 += 32 * kDecWarps) {   // uniform in the warp
    const int j = j0 + lane;
    const bool live = j < k1;
    // ---- this lane's K row and its columns of the 32 V rows, all requested up front so
    // that the whole step's bytes are in flight while the scores are formed
    uint4 kr[D / 8];
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8)
      kr[c8] = live ? __ldg(reinterpret_cast<const uint4*>(kh + (size_t)j * D + c8 * 8)) : make_uint4(0u, 0u, 0u, 0u);
    using VW = typename std::conditional<kCols == 2, unsigned int, uint2>::type;
    auto load_v = [&](int kk) -> VW {
      if (j0 + kk < k1) return __ldg(reinterpret_cast<const VW*>(vh + (size_t)(j0 + kk) * D + lane * kCols));
      if constexpr (kCols == 2) return 0u;
      else return make_uint2(0u, 0u);
    };
    VW vr[kVEarly ? 32 : 1];
    (void)vr;
    if constexpr (kVEarly) {
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) vr[kk] = load_v(kk);
    }
    float dot[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) dot[m] = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
      float kf[8];
      const uint32_t kw[4] = {kr[c8].x, kr[c8].y, kr[c8].z, kr[c8].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = unpack2<DT>(kw[c]);
        kf[2 * c] = f.x;
        kf[2 * c + 1] = f.y;
      }
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float4 qa = *reinterpret_cast<const float4*>(&sq[m][c8 * 8]);
        const float4 qb = *reinterpret_cast<const float4*>(&sq[m][c8 * 8 + 4]);
        dot[m] = fmaf(qa.x, kf[0], dot[m]);
        dot[m] = fmaf(qa.y, kf[1], dot[m]);
        dot[m] = fmaf(qa.z, kf[2], dot[m]);
        dot[m] = fmaf(qa.w, kf[3], dot[m]);
        dot[m] = fmaf(qb.x, kf[4], dot[m]);
        dot[m] = fmaf(qb.y, kf[5], dot[m]);
        dot[m] = fmaf(qb.z, kf[6], dot[m]);
        dot[m] = fmaf(qb.w, kf[7], dot[m]);
      }
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
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[m][c] *= a;
        mrow[m] = bm;
      }
      p[m] = x == -INFINITY ? 0.f : ex2_approx(x - mrow[m]);
      lrow[m] += p[m];
    }
#pragma unroll
    for (int m4 = 0; m4 < MR; m4 += 4) {
      if constexpr (MR >= 4)
        *reinterpret_cast<float4*>(pw + lane * MR + m4) = make_float4(p[m4], p[m4 + 1], p[m4 + 2], p[m4 + 3]);
    }
    if constexpr (MR < 4) {
#pragma unroll
      for (int m = 0; m < MR; ++m) pw[lane * MR + m] = p[m];
    }
    __syncwarp();
    // ---- O += P V: this lane's columns of the 32 V rows (rows past the range hold
    // zeros and have P = 0)
    auto pv_row = [&](int kk, VW vw) {
      float vf[kCols];
      if constexpr (kCols == 2) {
        const float2 f = unpack2<DT>(vw);
        vf[0] = f.x;
        vf[1] = f.y;
      } else {
        const float2 f0 = unpack2<DT>(vw.x), f1 = unpack2<DT>(vw.y);
        vf[0] = f0.x;
        vf[1] = f0.y;
        vf[2] = f1.x;
        vf[3] = f1.y;
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
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[m][c] = fmaf(pk[m], vf[c], acc[m][c]);
      }
    };
    if constexpr (kVEarly) {
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) pv_row(kk, vr[kk]);
    } else {
      const int nk = min(32, k1 - j0);
#pragma unroll 8
      for (int kk = 0; kk < nk; ++kk) pv_row(kk, load_v(kk));
    }
    __syncwarp();
  }

  // each warp: l = sum over lanes; O columns are already per lane
#pragma unroll
  for (int m = 0; m < MR; ++m) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lrow[m] += __shfl_xor_sync(0xffffffffu, lrow[m], off);
#pragma unroll
    for (int c = 0; c < kCols; ++c) sm_acc[warp][m][lane * kCols + c] = acc[m][c];
    if (lane == 0) {
      sm_m[warp][m] = mrow[m];
      sm_l[warp][m] = lrow[m];
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
      for (int c = 0; c < 8; ++c) a[c] += sm_acc[w][m][rr * 8 + c] * sc;
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

template <int DT, int MR>
__global__ void __launch_bounds__(kDecThreads, 1) decode_split_kernel_d64(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    float* __restrict__ opart, float* __restrict__ lpart, uint16_t* __restrict__ out, float* __restrict__ lse,
    int H, int Hkv, int Nq, int Nk, int M, int chunk, float scale_log2, int causal) {
  decode_split<64, DT, MR>(q, k, v, opart, lpart, out, lse, H, Hkv, Nq, Nk, M, chunk, scale_log2, causal);
}

template <int DT, int MR>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel_d128(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    float* __restrict__ opart, float* __restrict__ lpart, uint16_t* __restrict__ out, float* __restrict__ lse,
    int H, int Hkv, int Nq, int Nk, int M, int chunk, float scale_log2, int causal) {
  decode_split<128, DT, MR>(q, k, v, opart, lpart, out, lse, H, Hkv, Nq, Nk, M, chunk, scale_log2, causal);
}

// ---------------------------------------------------------------- TMA-fed split kernel
// The same split pass with K and V moved by the tensor memory accelerator: a producer
// warp streams the range's keys in stages of 32 rows (K and V, 64-column blocks with the
// 128-byte swizzle) through a ring of kDtStages stages in shared memory, and kDtWarps
// consumer warps take the stages in turn (stage s to warp s mod kDtWarps).  The bytes in
// flight no longer sit in registers, so one CTA per SM keeps the ring full, where the
// register-fed kernel was latency-bound.  Each consumer warp does exactly the
// register-fed kernel's step on its stage: one key per lane for the scores (a lane reads
// its K row, conflict-free in the swizzled layout), D/32 columns per lane for P V.
//
// Every ring slot belongs to one consumer warp (two slots per warp, used alternately), so
// a warp waits on a slot only after it has itself consumed the slot's previous use: a
// parity wait can then never be satisfied by a phase that is one use behind.
constexpr int kDtWarps = 6;
constexpr int kDtThreads = (kDtWarps + 1) * 32;
constexpr int kDtStages = 2 * kDtWarps;
// ring slot of stage s (the consuming warp's slot for its (s / kDtWarps)-th stage) and
// the use of that slot it is
__device__ __forceinline__ int dt_slot(int s) { return (s % kDtWarps) + kDtWarps * ((s / kDtWarps) & 1); }
__device__ __forceinline__ int dt_use(int s) { return (s / kDtWarps) >> 1; }

template <int D>
struct DtCfg {
  static constexpr int kBlock = 32 * 128;             // 32 rows x one 64-column block (128 bytes)
  static constexpr int kHalf = (D / 64) * kBlock;     // K, or V, of one stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kOffBar = kDtStages * kStage;
  static constexpr int kSmem = kOffBar + 2 * kDtStages * 8 + 1024;   // + alignment slack
};

template <int D, int DT, int MR>
__global__ void __launch_bounds__(kDtThreads, 1) decode_tma_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const uint16_t* __restrict__ q, float* __restrict__ opart, float* __restrict__ lpart,
    uint16_t* __restrict__ out, float* __restrict__ lse, int H, int Hkv, int Nq, int Nk, int M, int chunk,
    float scale_log2, int causal, unsigned int* err_word, uint64_t limit_ns) {
  using C = DtCfg<D>;
  constexpr int kCols = D / 32;                // output columns per lane
  __shared__ __align__(16) float sq[MR][D];    // query rows times scale*log2(e)
  __shared__ __align__(16) float sp[kDtWarps][32][MR];
  __shared__ float sm_m[kDtWarps][MR];
  __shared__ float sm_l[kDtWarps][MR];
  __shared__ int abort_flag;
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* ring = dsm_raw + ((1024u - (smem_u32(dsm_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::kOffBar);
  auto full = [&](int i) { return smem_u32(bars + i); };
  auto empty = [&](int i) { return smem_u32(bars + kDtStages + i); };

  const int split = blockIdx.x, S = gridDim.x;
  const int bhk = blockIdx.y, BHkv = gridDim.y;
  const int lane = threadIdx.x & 31;
  const int warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const int k0 = split * chunk;
  const int k1 = min(Nk, k0 + chunk);
  const int nst = (k1 - k0 + 31) / 32;         // stages of this range
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDtStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  grid_dep_wait();
  for (int i = threadIdx.x; i < MR * (D / 8); i += kDtThreads) {
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

  float mrow[MR], lrow[MR], acc[MR][kCols];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    mrow[m] = -INFINITY;
    lrow[m] = 0.f;   // this lane's share of l
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[m][c] = 0.f;
  }

  if (warp == kDtWarps) {
    // ---------------------------------------------------------- producer (one lane issues)
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    bool ok = true;
    int s = 0;
    for (; s < nst; ++s) {
      const int slot = dt_slot(s);
      if (s >= kDtStages && !wait_warp(empty(slot), (dt_use(s) - 1) & 1, ctl, 0x801)) {
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
      for (int t = (s > kDtStages ? s - kDtStages : 0); t < s; ++t)
        mbar_wait(full(dt_slot(t)), dt_use(t) & 1, drain, 0x8f1);
    }
  } else {
    // ---------------------------------------------------------- consumers
    int lim[MR];   // last key each query row sees (-1: a padding row sees none)
#pragma unroll
    for (int m = 0; m < MR; ++m) lim[m] = m < M ? (causal ? (m % Nq) + (Nk - Nq) : Nk - 1) : -1;
    float* pw = &sp[warp][0][0];
    for (int s = warp; s < nst; s += kDtWarps) {
      const int slot = dt_slot(s);
      if (!wait_warp(full(slot), dt_use(s) & 1, ctl, 0x802)) break;
      const uint8_t* kbuf = ring + slot * C::kStage;
      const uint8_t* vbuf = kbuf + C::kHalf;
      const int j0 = k0 + 32 * s;
      const int j = j0 + lane;
      const bool live = j < k1;
      float dot[MR];
#pragma unroll
      for (int m = 0; m < MR; ++m) dot[m] = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) {
        // this lane's key row, 16 bytes of it: block c8/8, swizzled unit (c8 % 8) ^ (row % 8)
        const uint4 kr = *reinterpret_cast<const uint4*>(kbuf + (c8 >> 3) * C::kBlock + lane * 128 +
                                                         (((c8 & 7) ^ (lane & 7)) << 4));
        float kf[8];
        const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = unpack2<DT>(kw[c]);
          kf[2 * c] = f.x;
          kf[2 * c + 1] = f.y;
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          const float4 qa = *reinterpret_cast<const float4*>(&sq[m][c8 * 8]);
          const float4 qb = *reinterpret_cast<const float4*>(&sq[m][c8 * 8 + 4]);
          dot[m] = fmaf(qa.x, kf[0], dot[m]);
          dot[m] = fmaf(qa.y, kf[1], dot[m]);
          dot[m] = fmaf(qa.z, kf[2], dot[m]);
          dot[m] = fmaf(qa.w, kf[3], dot[m]);
          dot[m] = fmaf(qb.x, kf[4], dot[m]);
          dot[m] = fmaf(qb.y, kf[5], dot[m]);
          dot[m] = fmaf(qb.z, kf[6], dot[m]);
          dot[m] = fmaf(qb.w, kf[7], dot[m]);
        }
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
#pragma unroll
          for (int c = 0; c < kCols; ++c) acc[m][c] *= a;
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
        float vf[kCols];
        if constexpr (kCols == 2) {
          const float2 f = unpack2<DT>(*reinterpret_cast<const uint32_t*>(vrow));
          vf[0] = f.x;
          vf[1] = f.y;
        } else {
          const uint2 w2 = *reinterpret_cast<const uint2*>(vrow);
          const float2 f0 = unpack2<DT>(w2.x), f1 = unpack2<DT>(w2.y);
          vf[0] = f0.x;
          vf[1] = f0.y;
          vf[2] = f1.x;
          vf[3] = f1.y;
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
#pragma unroll
          for (int c = 0; c < kCols; ++c) acc[m][c] = fmaf(pk[m], vf[c], acc[m][c]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(slot));
    }
  }
  // every stage has been read (or the ring drained): its memory now holds the warps' sums
  __syncthreads();
  float* sm_acc = reinterpret_cast<float*>(ring);   // [kDtWarps][MR][D]
  if (warp < kDtWarps) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lrow[m] += __shfl_xor_sync(0xffffffffu, lrow[m], off);
#pragma unroll
      for (int c = 0; c < kCols; ++c) sm_acc[(warp * MR + m) * D + lane * kCols + c] = acc[m][c];
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
    for (int w = 0; w < kDtWarps; ++w) mx = fmaxf(mx, sm_m[w][m]);
    float lsum = 0.f, a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kDtWarps; ++w) {
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
  cudaError_t e;
  if (a.tma) {
    auto kern = decode_tma_kernel<D, DT, MR>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DtCfg<D>::kSmem);
    if (e != cudaSuccess) return e;
    e = launch_overlapped(kern, dim3(a.S, a.BHkv), kDtThreads, DtCfg<D>::kSmem, stream, a.tm_k, a.tm_v,
                          static_cast<const uint16_t*>(a.q), a.opart, a.lpart, static_cast<uint16_t*>(a.o), a.lse,
                          a.H, a.Hkv, a.Nq, a.Nk, a.M, a.chunk, a.scale_log2, a.causal, a.err_word, a.limit_ns);
  } else {
    auto kern = D == 64 ? decode_split_kernel_d64<DT, MR> : decode_split_kernel_d128<DT, MR>;
    e = launch_overlapped(kern, dim3(a.S, a.BHkv), kDecThreads, 0, stream, static_cast<const uint16_t*>(a.q),
                          static_cast<const uint16_t*>(a.k), static_cast<const uint16_t*>(a.v), a.opart, a.lpart,
                          static_cast<uint16_t*>(a.o), a.lse, a.H, a.Hkv, a.Nq, a.Nk, a.M, a.chunk, a.scale_log2,
                          a.causal);
  }
  if (e != cudaSuccess || a.S == 1) return e;
  const long long threads = (long long)a.BHkv * a.M * (D / 8);
  return launch_overlapped(decode_merge_kernel<D, DT>, dim3((unsigned)((threads + 255) / 256)), 256, 0, stream,
                           static_cast<const float*>(a.opart), static_cast<const float*>(a.lpart),
                           static_cast<uint16_t*>(a.o), a.lse, a.BHkv, a.H, a.Hkv, a.Nq, a.M, a.S);
}

// Resident split-kernel CTAs per SM (registers and shared memory decide), 0 on error.
template <int D, int DT, int MR>
int ctas_per_sm_t() {
  auto kern = D == 64 ? decode_split_kernel_d64<DT, MR> : decode_split_kernel_d128<DT, MR>;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecThreads, 0) != cudaSuccess) return 0;
  return n;
}

template <int D, int DT>
int ctas_per_sm_m(int M) {
  if (M <= 1) return ctas_per_sm_t<D, DT, 1>();
  if (M <= 2) return ctas_per_sm_t<D, DT, 2>();
  if (M <= 4) return ctas_per_sm_t<D, DT, 4>();
  return ctas_per_sm_t<D, DT, 8>();
}

template <int D, int DT>
cudaError_t launch_decode_m(const DecArgs& a, cudaStream_t stream) {
  if (a.M <= 1) return launch_decode_t<D, DT, 1>(a, stream);
  if (a.M <= 2) return launch_decode_t<D, DT, 2>(a, stream);
  if (a.M <= 4) return launch_decode_t<D, DT, 4>(a, stream);
  return launch_decode_t<D, DT, 8>(a, stream);
}

}  // namespace

int decode_keys_per_step(int d) { return 32 * kDecWarps + 0 * d; }

int decode_ctas_per_sm(int d, int dtype, int M) {
  // one entry per (d, dtype, row bucket); the answer depends only on the compiled kernel
  static std::atomic<int> cache[16];
  const int bucket = M <= 1 ? 0 : M <= 2 ? 1 : M <= 4 ? 2 : 3;
  const int key = ((d == 128 ? 2 : 0) | (dtype == 1 ? 1 : 0)) * 4 + bucket;
  int n = cache[key].load(std::memory_order_relaxed);
  if (n > 0) return n;
  switch (key >> 2) {
    case 0: n = ctas_per_sm_m<64, 0>(M); break;
    case 1: n = ctas_per_sm_m<64, 1>(M); break;
    case 2: n = ctas_per_sm_m<128, 0>(M); break;
    default: n = ctas_per_sm_m<128, 1>(M); break;
  }
  if (n > 0) cache[key].store(n, std::memory_order_relaxed);
  return n;
}

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
