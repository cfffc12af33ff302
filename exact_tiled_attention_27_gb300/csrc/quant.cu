// quant.cu -- E4M3 block quantization for the FP8 forward (fa_quantize_fp8).
//
// The FP8 variant of the "Flash Attention" chapter (mlx.void.app), section
// "FlashAttention-3——重叠与低精度": an E4M3 number has 256 bit patterns and a largest
// value of 448, so everything rests on the scale that maps the data onto that grid.
// Block quantization gives every block its own scale, so an outlier spoils only its own
// block; incoherent processing multiplies Q and K by one fixed random rotation before
// rounding, spreading an outlier over every dimension without changing any dot product.
//
// One (head, 128-row block) per CTA and one row per thread.  With one scale per block
// a single launch does everything (quant_codes_kernel<FUSED>): the block's rows
// (rotated when signs are given) stay in registers while the CTA reduces their largest
// magnitude, then scale = amax / 448 (1 when amax = 0) and code = E4M3(x * (1 / scale)),
// written row-major, or transposed to (d, Nt) rows of keys for the V^T operand of the
// P.V product.  One scale per tensor needs the head's largest magnitude first, so that
// mode runs three launches: quant_amax_kernel (block amax into scales[]),
// quant_scale_kernel (the head's amax / 448 into every block), quant_codes_kernel.
// The rotation is x -> x diag(signs) H / sqrt(d) with H the Sylvester-Hadamard matrix,
// evaluated by the radix-2 butterflies h = 1, 2, 4, ... in float32.  Every rounding
// step is a fixed round-to-nearest operation, so the codes are reproducible bit for bit.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kQRows = 128;
constexpr float kE4M3Max = 448.0f;

// Row `row` of x as float32, rotated when ROT.
template <int D, int DT, bool ROT>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ x, size_t row, const float* __restrict__ signs,
                                         float (&y)[D]) {
  const uint4* src = reinterpret_cast<const uint4*>(x + row * D);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 w = __ldg(src + c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack2<DT>(ws[i]);
      y[8 * c + 2 * i] = f.x;
      y[8 * c + 2 * i + 1] = f.y;
    }
  }
  if constexpr (ROT) {
#pragma unroll
    for (int i = 0; i < D; ++i) y[i] = __fmul_rn(y[i], __ldg(signs + i));   // exact: signs are +-1
#pragma unroll
    for (int h = 1; h < D; h <<= 1) {
#pragma unroll
      for (int i = 0; i < D; ++i) {
        if ((i & h) == 0) {
          const float a = y[i], b = y[i + h];
          y[i] = __fadd_rn(a, b);
          y[i + h] = __fsub_rn(a, b);
        }
      }
    }
    const float c = (D == 64) ? 0.125f : 0.08838834764831845f;   // fl32(1 / sqrt(d))
#pragma unroll
    for (int i = 0; i < D; ++i) y[i] = __fmul_rn(y[i], c);
  }
}

// The block's largest magnitude, reduced over the CTA and returned to every thread.
__device__ __forceinline__ float block_amax(float m) {
  __shared__ float part[kQRows / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  float b = part[0];
#pragma unroll
  for (int w = 1; w < kQRows / 32; ++w) b = fmaxf(b, part[w]);
  return b;
}

template <int D, int DT, bool ROT>
__global__ void __launch_bounds__(kQRows) quant_amax_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ signs,
                                                            float* __restrict__ amax, int N, int nb) {
  const int bh = blockIdx.x / nb;
  const int blk = blockIdx.x - bh * nb;
  const int r = blk * kQRows + threadIdx.x;
  float m = 0.f;
  if (r < N) {
    float y[D];
    load_row<D, DT, ROT>(x, (size_t)bh * N + r, signs, y);
#pragma unroll
    for (int i = 0; i < D; ++i) m = fmaxf(m, fabsf(y[i]));
  }
  const float b = block_amax(m);
  if (threadIdx.x == 0) amax[blockIdx.x] = b;
}

// One warp per head; turns the block amax values into scales in place.
__global__ void __launch_bounds__(256) quant_scale_kernel(float* __restrict__ scales, int BH, int nb, int per_tensor) {
  const int head = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (head >= BH) return;
  float* s = scales + (size_t)head * nb;
  float hm = 0.f;
  if (per_tensor) {
    for (int j = lane; j < nb; j += 32) hm = fmaxf(hm, s[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, o));
  }
  for (int j = lane; j < nb; j += 32) {
    const float a = per_tensor ? hm : s[j];
    s[j] = a > 0.f ? __fdiv_rn(a, kE4M3Max) : 1.0f;
  }
}

// FUSED: compute and write the block's scale here (one scale per block); otherwise read
// it from scales[].
template <int D, int DT, bool ROT, bool TR, bool FUSED>
__global__ void __launch_bounds__(kQRows) quant_codes_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ signs,
                                                             float* __restrict__ scales,
                                                             uint8_t* __restrict__ x8, int N, int nb, int Nt) {
  const int bh = blockIdx.x / nb;
  const int blk = blockIdx.x - bh * nb;
  const int r = blk * kQRows + threadIdx.x;
  float y[D];
  if (r < N) load_row<D, DT, ROT>(x, (size_t)bh * N + r, signs, y);
  float scale;
  if constexpr (FUSED) {
    float m = 0.f;
    if (r < N) {
#pragma unroll
      for (int i = 0; i < D; ++i) m = fmaxf(m, fabsf(y[i]));
    }
    const float amax = block_amax(m);
    scale = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
    if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  } else {
    scale = scales[blockIdx.x];
  }
  const float inv = __frcp_rn(scale);
  uint32_t w[D / 4];
  if (r < N) {
#pragma unroll
    for (int q = 0; q < D / 4; ++q)
      w[q] = pack4_e4m3(__fmul_rn(y[4 * q], inv), __fmul_rn(y[4 * q + 1], inv), __fmul_rn(y[4 * q + 2], inv),
                        __fmul_rn(y[4 * q + 3], inv));
  } else {
#pragma unroll
    for (int q = 0; q < D / 4; ++q) w[q] = 0u;   // keys in [N, Nt) of the transposed layout read as +0
  }
  if constexpr (!TR) {
    if (r < N) {
      uint4* dst = reinterpret_cast<uint4*>(x8 + ((size_t)bh * N + r) * D);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
  } else {
    // the block's codes, transposed in shared memory: column c of the block is row c
    // (128 keys) of V^T
    __shared__ __align__(16) uint8_t t[D * kQRows];
#pragma unroll
    for (int q = 0; q < D / 4; ++q)
#pragma unroll
      for (int b = 0; b < 4; ++b) t[(4 * q + b) * kQRows + threadIdx.x] = (uint8_t)(w[q] >> (8 * b));
    __syncthreads();
    const int k0 = blk * kQRows;
    const int chunks = min(kQRows, Nt - k0) / 16;   // Nt is a multiple of 16 and k0 < N <= Nt
    for (int i = threadIdx.x; i < D * (kQRows / 16); i += kQRows) {
      const int c = i / (kQRows / 16), u = i % (kQRows / 16);
      if (u < chunks)
        *reinterpret_cast<uint4*>(x8 + ((size_t)bh * D + c) * Nt + k0 + u * 16) =
            *reinterpret_cast<const uint4*>(t + c * kQRows + u * 16);
    }
  }
}

template <int D, int DT, bool ROT>
cudaError_t launch_quant_t(const QuantArgs& a, cudaStream_t stream) {
  const int nb = (a.N + kQRows - 1) / kQRows;
  const unsigned grid = (unsigned)((size_t)a.BH * nb);
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  uint8_t* x8 = static_cast<uint8_t*>(a.x8);
  if (!a.per_tensor) {
    if (a.transpose)
      quant_codes_kernel<D, DT, ROT, true, true><<<grid, kQRows, 0, stream>>>(x, a.signs, a.scales, x8, a.N, nb, a.Nt);
    else
      quant_codes_kernel<D, DT, ROT, false, true><<<grid, kQRows, 0, stream>>>(x, a.signs, a.scales, x8, a.N, nb, a.Nt);
    return cudaGetLastError();
  }
  quant_amax_kernel<D, DT, ROT><<<grid, kQRows, 0, stream>>>(x, a.signs, a.scales, a.N, nb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned sgrid = (unsigned)(((size_t)a.BH * 32 + 255) / 256);
  quant_scale_kernel<<<sgrid, 256, 0, stream>>>(a.scales, a.BH, nb, a.per_tensor);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.transpose)
    quant_codes_kernel<D, DT, ROT, true, false><<<grid, kQRows, 0, stream>>>(x, a.signs, a.scales, x8, a.N, nb, a.Nt);
  else
    quant_codes_kernel<D, DT, ROT, false, false><<<grid, kQRows, 0, stream>>>(x, a.signs, a.scales, x8, a.N, nb, a.Nt);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quant_d(const QuantArgs& a, cudaStream_t stream) {
  const bool rot = a.signs != nullptr;
  if (a.dtype == 1) return rot ? launch_quant_t<D, 1, true>(a, stream) : launch_quant_t<D, 1, false>(a, stream);
  return rot ? launch_quant_t<D, 0, true>(a, stream) : launch_quant_t<D, 0, false>(a, stream);
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_quant_d<128>(a, stream) : launch_quant_d<64>(a, stream);
}

}  // namespace fa
