// fwd_fp8.cu -- FP8 (E4M3) forward of exact tiled attention for sm_103a.
//
// The FP8 lever of the "Flash Attention" chapter (mlx.void.app), section
// "FlashAttention-3——重叠与低精度": Q, K and V are E4M3 codes with one scale per
// 128-row block (block quantization; fa_quantize_fp8 makes them, optionally after
// multiplying Q and K by a fixed random rotation), and both matrix products run on the
// 8-bit tensor-core path (tcgen05.mma kind::f8f6f4, 32 elements of K per instruction,
// fp32 accumulation) at twice the 16-bit rate.
//
// The structure is the 16-bit forward's (fwd.cu): persistent CTAs over work tiles of
// two 128-row query blocks, warps 0-7 two softmax warpgroups (one thread per query
// row), warp 8 the TMA producer, warp 9 the MMA issuer, S_t in tensor memory and the
// unnormalised O_t there too.  What differs:
//
//   * operands: Q and K tiles are 128 rows of d bytes (64-byte swizzle at d = 64,
//     128-byte at d = 128).  V is stored transposed, V^T with one row of keys per
//     channel, so that the B operand of P.V is K-major like every other 8-bit operand.
//     P is the A operand from tensor memory, four E4M3 codes per column over the first
//     32 columns of S_t (S_t(j+1) is issued after P_t(j).V by the same thread, and the
//     tensor core runs them in that order).
//   * scales: block j of K scales S by sk_j, and the query block by sq, so the exponent
//     uses c_j = scale * log2(e) * sq * sk_j.  The scale sv_j of V block j is folded
//     into that block's probabilities before they are rounded: the kernel works with
//     y = s c_j + log2(sv_j), so P.V needs no per-block rescale of O, and the running
//     sum l adds the same probabilities divided by sv_j.
//   * P: rounded to E4M3 and written back to tensor memory.  The running maximum M
//     only moves when a row maximum exceeds it by more than 4 (base 2), and P is
//     formed as 2^(y - M + 4), so
//     P <= 2^8 stays below E4M3's 448 and entries down to 2^-13 of a row's largest
//     stay representable; O is rescaled only on the rare steps where M moves.
//   * sums: l adds the unrounded P (lse = (M - 4 + log2 l) ln 2); lr, which divides O,
//     adds them too but takes each block's largest P as rounded to E4M3.  A row
//     dominated by one key is then normalised by the weight P.V actually used, and its
//     O does not carry that weight's rounding error (up to 2^-4).
#include <cuda_fp16.h>

#include "fwd_tiles.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kF8Threads = 384;
constexpr int kF8LaunchRegs = 168;
constexpr int kF8SoftmaxRegs = 216;
constexpr int kF8OtherRegs = 64;
static_assert((2 * kF8SoftmaxRegs + kF8OtherRegs) * 128 <= kF8LaunchRegs * kF8Threads,
              "register split exceeds the launch");
constexpr float kRescaleTau = 4.0f;                // M moves when a row maximum exceeds it by more than this
constexpr float kPHeadroom = 8.0f - kRescaleTau;   // P = 2^(y - M + 4) <= 2^8 < 448

template <int D>
struct F8Cfg {
  static constexpr int kTileBytes = kTileRows * D;          // Q, K: 128 rows x d bytes; V^T: d rows x 128 bytes
  static constexpr int kQBufs = (D == 64) ? 2 : 1;
  static constexpr int kStages = (D == 64) ? 8 : 6;
  static constexpr int kOffQ = 0;                           // [kQBufs][2 sub-tiles]
  static constexpr int kOffK = kOffQ + kQBufs * 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = kQFull + kQBufs;
  static constexpr int kKFull = kQEmpty + kQBufs;
  static constexpr int kVFull = kKFull + kStages;
  static constexpr int kKVEmpty = kVFull + kStages;
  static constexpr int kSFull = kKVEmpty + kStages;         // [2]
  static constexpr int kPHalf = kSFull + 2;                 // [2] codes of the first 64 keys written
  static constexpr int kPFull = kPHalf + 2;                 // [2]
  static constexpr int kOFull = kPFull + 2;                 // [2]
  static constexpr int kOEmpty = kOFull + 2;                // [2]
  static constexpr int kDrain = kOEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  // P_t (E4M3, four per column) occupies the first 32 columns of S_t
  __host__ __device__ static constexpr uint32_t tm_s(int t) { return t * 128; }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256 + t * 128; }
};

// K-major descriptor of a 128-row tile of d-byte rows, advanced to byte `k` of the row
template <int D>
__device__ __forceinline__ uint64_t rows_desc(uint32_t base, int k) {
  if constexpr (D == 64)
    return sdesc_sw64(base + k, 512);
  else
    return sdesc_sw128(base + k, 16, 1024);
}

template <int D, int DT, bool CAUSAL>
__global__ void __launch_bounds__(kF8Threads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const float* __restrict__ q_scale,
                   const float* __restrict__ k_scale, const float* __restrict__ v_scale, uint16_t* __restrict__ out,
                   float* __restrict__ lse, int BH, int N, float scale_log2, int pairing, unsigned int* err_word,
                   uint64_t limit_ns) {
  using C = F8Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
  const int nqb = (N + kTileRows - 1) / kTileRows;
  const int ntiles = forward_tiles(BH, nqb, pairing);

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
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(bar(C::kKFull + i), 1);
      mbar_init(bar(C::kVFull + i), 1);
      mbar_init(bar(C::kKVEmpty + i), 1);
    }
    mbar_init(bar(C::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
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
  grid_dep_wait();

  if (warp >= 8) regs_dec<kF8OtherRegs>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (whole warp; one lane issues)
    if (elect_one()) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_vt);
    }
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (int k = 0, tile = persistent_tile(0); ok && tile < ntiles; tile = persistent_tile(++k), ++it) {
      const TileInfo ti = decode_tile<0>(tile, BH, 1, 1, N, N, CAUSAL, pairing);
      const int qbuf = it % C::kQBufs;
      if (it >= C::kQBufs && !wait_warp(bar(C::kQEmpty + qbuf), ((it / C::kQBufs) - 1) & 1, ctl, 0x901)) {
        ok = false;
        break;
      }
      const int nsub = ti.n1 > 0 ? 2 : 1;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(C::kQFull + qbuf), nsub * C::kTileBytes);
        for (int t = 0; t < nsub; ++t)
          tma_load_3d(smem_u32(smem + C::kOffQ + (qbuf * 2 + t) * C::kTileBytes), &tm_q, bar(C::kQFull + qbuf), 0,
                      (t == 0 ? ti.qb0 : ti.qb1) * kTileRows, ti.bh);
      }
      __syncwarp();
      for (int j = 0; j < ti.nkv; ++j, ++g) {
        const int st = g % C::kStages;
        if (g >= (uint32_t)C::kStages &&
            !wait_warp(bar(C::kKVEmpty + st), ((g / C::kStages) - 1) & 1, ctl, 0x902)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::kKFull + st), C::kTileBytes);
          tma_load_3d(smem_u32(smem + C::kOffK + st * C::kTileBytes), &tm_k, bar(C::kKFull + st), 0, j * kTileRows,
                      ti.bh);
          mbar_arrive_expect_tx(bar(C::kVFull + st), C::kTileBytes);
          tma_load_3d(smem_u32(smem + C::kOffV + st * C::kTileBytes), &tm_vt, bar(C::kVFull + st), j * kTileRows, 0,
                      ti.bh);
        }
        __syncwarp();
      }
    }
    if (!ok) {   // every copy already issued must land before the CTA exits
      for (int st = 0; st < C::kStages; ++st) {
        if (g > (uint32_t)st) {
          const uint32_t last = g - 1 - ((g - 1 - st) % C::kStages);
          mbar_wait(bar(C::kKFull + st), (last / C::kStages) & 1, drain, 0x9f1);
          mbar_wait(bar(C::kVFull + st), (last / C::kStages) & 1, drain, 0x9f2);
        }
      }
      for (int b = 0; b < C::kQBufs; ++b) {
        if (it > b) {
          const int last = it - 1 - ((it - 1 - b) % C::kQBufs);
          mbar_wait(bar(C::kQFull + b), (last / C::kQBufs) & 1, drain, 0x9f3);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (whole warp; one lane issues)
    constexpr uint32_t idesc_s = idesc_e4m3(128, 128);
    constexpr uint32_t idesc_o = idesc_e4m3(128, D);
    uint32_t g = 0;
    int it = 0;
    uint32_t c[2] = {0, 0};
    uint32_t e[2] = {0, 0};
    bool ok = true;
    auto issue_s = [&](int t, uint32_t qbase, uint32_t kbase) {
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk)   // S = Q K^T: A = Q, B = K, both K-major; 32 codes per step
        umma_ss_f8(tmem + C::tm_s(t), rows_desc<D>(qbase, kk * 32), rows_desc<D>(kbase, kk * 32), idesc_s,
                   kk > 0 ? 1u : 0u);
    };
    for (int k = 0, tile = persistent_tile(0); ok && tile < ntiles; tile = persistent_tile(++k), ++it) {
      const TileInfo ti = decode_tile<0>(tile, BH, 1, 1, N, N, CAUSAL, pairing);
      const int n[2] = {ti.n0, ti.n1};
      const int qbuf = it % C::kQBufs;
      const uint32_t qbase0 = smem_u32(smem + C::kOffQ + (qbuf * 2) * C::kTileBytes);
      if (!wait_warp(bar(C::kQFull + qbuf), (it / C::kQBufs) & 1, ctl, 0xa01)) break;
      if (!wait_warp(bar(C::kKFull + g % C::kStages), (g / C::kStages) & 1, ctl, 0xa02)) break;
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
        if (j + 1 < ti.nkv && !wait_warp(bar(C::kKFull + stn), ((gj + 1) / C::kStages) & 1, ctl, 0xa03)) {
          ok = false;
          break;
        }
        if (!wait_warp(bar(C::kVFull + st), (gj / C::kStages) & 1, ctl, 0xa04)) {
          ok = false;
          break;
        }
        const uint32_t vbase = smem_u32(smem + C::kOffV + st * C::kTileBytes);
        const uint32_t knext = smem_u32(smem + C::kOffK + stn * C::kTileBytes);
        // O += P V for keys [32*kk0, 32*kk1): A = P from tensor memory (32 keys = 8
        // columns), B = V^T (d x keys)
        auto issue_pv = [&](int t, int kk0, int kk1) {
#pragma unroll
          for (int kk = kk0; kk < kk1; ++kk)
            umma_ts_f8(tmem + C::tm_o(t), tmem + C::tm_s(t) + kk * 8, sdesc_sw128(vbase + kk * 32, 16, 1024),
                       idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        };
        for (int t = 0; t < 2; ++t) {
          if (j >= n[t]) continue;
          // the first 64 keys' codes are in tensor memory: their product overlaps the
          // softmax's exponentials of the other 64
          if (!wait_warp(bar(C::kPHalf + t), c[t] & 1, ctl, 0xa05) ||
              (j == 0 && e[t] > 0 && !wait_warp(bar(C::kOEmpty + t), (e[t] - 1) & 1, ctl, 0xa06))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) issue_pv(t, 0, kTileRows / 64);
          __syncwarp();
          if (!wait_warp(bar(C::kPFull + t), c[t] & 1, ctl, 0xa07)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, kTileRows / 64, kTileRows / 32);
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
    if (elect_one()) umma_commit(bar(C::kDrain));
    __syncwarp();
    mbar_wait(bar(C::kDrain), 0, drain, 0xaf1);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<kF8SoftmaxRegs>();
    const int t = warp >> 2;
    const int tid = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + C::tm_s(t);
    const uint32_t o_addr = tmem + lane_base + C::tm_o(t);
    uint32_t c = 0;
    uint32_t e = 0;
    for (int k = 0, tile = persistent_tile(0); tile < ntiles; tile = persistent_tile(++k)) {
      const TileInfo ti = decode_tile<0>(tile, BH, 1, 1, N, N, CAUSAL, pairing);
      const int n = t == 0 ? ti.n0 : ti.n1;
      if (n == 0) continue;
      const int qb = t == 0 ? ti.qb0 : ti.qb1;
      const int row = qb * kTileRows + tid;
      const int lim_row = CAUSAL ? min(N - 1, row) : (N - 1);
      const size_t sbase = (size_t)ti.bh * nqb;
      const float cq = scale_log2 * __ldg(q_scale + sbase + qb);
      float sk = __ldg(k_scale + sbase);   // block 0; the next block's scales are fetched a step ahead
      float sv = __ldg(v_scale + sbase);
      float m = -INFINITY;
      float l = 0.f;    // sum of P as computed: lse
      float lr = 0.f;   // the same with each block's largest P as rounded: divides O
      bool ok = true;
      for (int j = 0; j < n; ++j, ++c) {
        const float cj = cq * sk;
        const float vj = lg2_approx(sv);
        if (j + 1 < n) {
          sk = __ldg(k_scale + sbase + j + 1);
          sv = __ldg(v_scale + sbase + j + 1);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + t), c & 1, ctl, 0xb01))) {
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
        const int kbase = j * kTileRows;
        if ((kbase + kTileRows > N) || (CAUSAL && j == qb)) {
#pragma unroll
          for (int q = 0; q < 128; ++q)
            if (kbase + q > lim_row) s[q] = -INFINITY;
        }
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
        const float ymax = mx * cj + vj;
        const float m_new = (ymax > m + kRescaleTau) ? ymax : m;
        const float alpha = (m_new == m) ? 1.0f : ex2_approx(m - m_new);   // 0 on the first block
        const uint64_t c2 = f2_pack(cj, cj);
        const float off = vj + kPHeadroom - m_new;
        const uint64_t off2 = f2_pack(off, off);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          // O holds every earlier P.V (committed before this S): bring it to the new
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
        }
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P (four E4M3 codes per column) over the first 32 columns of S_t, in two halves of
        // 64 keys, each handed to the MMA warp as soon as it is in tensor memory
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int qq = hf * 16 + q;
            float x0, x1, x2, x3;
            f2_unpack(ffma2(f2_pack(s[4 * qq], s[4 * qq + 1]), c2, off2), x0, x1);
            f2_unpack(ffma2(f2_pack(s[4 * qq + 2], s[4 * qq + 3]), c2, off2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc[q & 3] = fadd2(acc[q & 3], fadd2(f2_pack(p0, p1), f2_pack(p2, p3)));
            pk[q] = pack4_e4m3(p0, p1, p2, p3);
          }
          tmem_st16(s_addr + hf * 16, pk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(hf == 0 ? C::kPHalf + t : C::kPFull + t));
        }
        float a0, a1, b0, b1;
        f2_unpack(fadd2(acc[0], acc[1]), a0, a1);
        f2_unpack(fadd2(acc[2], acc[3]), b0, b1);
        const float rowsum = (a0 + a1) + (b0 + b1);
        const float pmax = ex2_approx(fmaf(mx, cj, off));   // the block's largest P, bit for bit
        const float inv_sv = ex2_approx(-vj);
        l = l * alpha + rowsum * inv_sv;
        lr = lr * alpha + (rowsum + (round_e4m3(pmax) - pmax)) * inv_sv;
        m = m_new;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::kOFull + t), e & 1, ctl, 0xb03))) break;
      ++e;
      tc_fence_after();
      const float inv_l = 1.0f / lr;
      uint8_t* orow = reinterpret_cast<uint8_t*>(out) + ((size_t)ti.bh * N + row) * (D * 2);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t orr[32];
        tmem_ld32(o_addr + q * 32, orr);
        tmem_ld_wait();
        reg_fence<32>(orr);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<DT>(__uint_as_float(orr[2 * i]) * inv_l, __uint_as_float(orr[2 * i + 1]) * inv_l);
        if (row < N) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_global_v4(orow + q * 64 + i * 16, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row < N) lse[(size_t)ti.bh * N + row] = (m - kPHeadroom + lg2_approx(l)) * 0.69314718055994530942f;
      tc_fence_before();
      mbar_arrive(bar(C::kOEmpty + t));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int DT, bool CAUSAL>
cudaError_t launch_fp8_t(const FwdF8Args& a, cudaStream_t stream) {
  using C = F8Cfg<D>;
  auto kern = fwd_fp8_kernel<D, DT, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * kF8Threads < (2 * kF8SoftmaxRegs + kF8OtherRegs) * 128) return cudaErrorInvalidConfiguration;
  int grid = 0;
  const int pairing = choose_pairing(a.BH, a.N, a.N, CAUSAL, true, true, a.num_sms, &grid);
  return launch_overlapped(kern, grid, kF8Threads, C::kSmemBytes, stream, a.tm_q, a.tm_k, a.tm_vt, a.q_scale,
                           a.k_scale, a.v_scale, static_cast<uint16_t*>(a.o), a.lse, a.BH, a.N, a.scale_log2,
                           pairing, a.err_word, a.limit_ns);
}

}  // namespace

cudaError_t launch_fwd_fp8(const FwdF8Args& a, cudaStream_t stream) {
  const int key = (a.d == 128 ? 4 : 0) | (a.dtype == 1 ? 2 : 0) | (a.causal ? 1 : 0);
  switch (key) {
    case 0: return launch_fp8_t<64, 0, false>(a, stream);
    case 1: return launch_fp8_t<64, 0, true>(a, stream);
    case 2: return launch_fp8_t<64, 1, false>(a, stream);
    case 3: return launch_fp8_t<64, 1, true>(a, stream);
    case 4: return launch_fp8_t<128, 0, false>(a, stream);
    case 5: return launch_fp8_t<128, 0, true>(a, stream);
    case 6: return launch_fp8_t<128, 1, false>(a, stream);
    default: return launch_fp8_t<128, 1, true>(a, stream);
  }
}

}  // namespace fa
