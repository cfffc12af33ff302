// fwd_tiles.cuh -- the work-tile schedule shared by the forward kernels (16-bit and
// FP8): which query blocks a persistent CTA takes next and which key/value blocks
// each of them visits.
//
// A work tile is one (batch*head) and two 128-row query blocks ("sub-tiles") that
// share every key/value block loaded for them.  Tiles are walked by the persistent
// CTAs in snake order (persistent_tile), heaviest causal tiles first, following the
// "FlashAttention-2" section of the "Flash Attention" chapter (mlx.void.app): the
// sequence is split into query blocks across the whole chip, and tiles wholly above
// the causal diagonal are skipped.
#pragma once

#include <algorithm>
#include <vector>

#include "internal.h"

namespace fa {
namespace {

constexpr int kTileRows = 128;   // query rows per sub-tile and keys per key/value block

struct TileInfo {
  int bh, kvh, qb0, qb1, n0, n1, nkv;
  bool has1;   // the second query block exists (it may still see no key)
  bool split;  // pairing 3: both sub-tiles take query block qb0, sub-tile 1 from key block koff1
  int koff1;
};

// Key/value blocks visible to query block qb: all of them without the causal mask;
// with it, up to the last key the block's last row may see.  The causal mask is
// aligned bottom-right: key j is visible to query i iff j <= i + (Nk - Nq), which is
// the square mask when Nq = Nk.  0 when no row of the block sees any key.
__host__ __device__ __forceinline__ int visible_kv_blocks(int qb, int Nq, int Nk, bool causal) {
  const int nkb = (Nk + kTileRows - 1) / kTileRows;
  if (!causal) return nkb;
  const int last_row = min(Nq - 1, qb * kTileRows + kTileRows - 1);
  const long long last_key = (long long)last_row + (Nk - Nq);
  if (last_key < 0) return 0;
  const int n = (int)(last_key / kTileRows) + 1;
  return n < nkb ? n : nkb;
}

// Work tile `tile` -> head, the two query blocks and their key/value block counts
// (n1 = 0 when there is no second block).  Three pairings of the query blocks:
//   0 adjacent  (2p, 2p+1): the two sub-tiles share every key/value block; pairs are
//               numbered heaviest first under the causal mask.
//   1 balanced  (i, nqb-1-i): under the causal mask every pair costs nqb+1 blocks, which
//               evens out the work when there are only about as many pairs as SMs.
//   2 single    one query block per tile, heaviest first: for launches with fewer pairs
//               than SMs, so that every SM works and a lone softmax warpgroup runs
//               without the other's contention.
//   3 split     single query blocks as in 2, with the block's keys cut in two: sub-tile 0
//               takes the first ceil(n/2) key blocks, sub-tile 1 the rest (koff1 on), and
//               the two partial results are merged at the end (16-bit forward, d = 64).
// MODE: 0 plain (Nq = Nk, one key/value head per query head), 1 general (fa_fwd_cross),
// 2 butterfly block pattern (fa_fwd_sparse).
template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(int tile, int BH, int H, int G, int Nq, int Nk, bool causal,
                                                int pairing) {
  const int nqb = (Nq + kTileRows - 1) / kTileRows;
  const int npairs = (nqb + 1) >> 1;
  TileInfo ti;
  const int r = tile / BH;
  ti.bh = tile - r * BH;
  ti.kvh = MODE == 1 ? (ti.bh / H) * (H / G) + (ti.bh % H) / G : ti.bh;
  if (pairing >= 2) {
    ti.qb0 = nqb - 1 - r;
    ti.qb1 = nqb;   // none
  } else if (pairing == 1) {
    ti.qb0 = r;
    ti.qb1 = nqb - 1 - r;
  } else {
    ti.qb0 = 2 * (npairs - 1 - r);   // r = 0: the last (heaviest, causal) pair of every head
    ti.qb1 = ti.qb0 + 1;
  }
  ti.has1 = ti.qb1 < nqb && ti.qb1 != ti.qb0;
  if constexpr (MODE == 1) {
    ti.n0 = visible_kv_blocks(ti.qb0, Nq, Nk, causal);
    ti.n1 = ti.has1 ? visible_kv_blocks(ti.qb1, Nq, Nk, causal) : 0;
  } else if constexpr (MODE == 2) {
    // both query blocks of pair p = qb0/2 walk the key blocks of p's linked pairs; under
    // the causal mask the list ends with block qb1, which query block qb0 does not see
    const int n = bfly_blocks(ti.qb0 >> 1, npairs, nqb, causal ? -1 : 0, 0);
    ti.n1 = ti.has1 ? n : 0;
    ti.n0 = (causal && ti.has1) ? n - 1 : n;
  } else {   // Nq = Nk: block qb sees blocks 0..qb under the causal mask
    ti.n0 = causal ? ti.qb0 + 1 : nqb;
    ti.n1 = ti.has1 ? (causal ? ti.qb1 + 1 : nqb) : 0;
  }
  ti.split = false;
  ti.koff1 = 0;
  if (pairing == 3) {
    const int n = ti.n0;
    ti.n0 = (n + 1) >> 1;
    ti.n1 = n - ti.n0;
    ti.qb1 = ti.qb0;
    ti.koff1 = ti.n0;
    ti.split = true;
  }
  ti.nkv = ti.n0 > ti.n1 ? ti.n0 : ti.n1;
  return ti;
}

// Causal pairing choice: simulate the snake schedule of both pairings over `grid`
// CTAs and keep the one whose busiest CTA has less work (adjacent on ties, since its
// sub-tiles share more key/value loads).  With many tiles per CTA both balance well,
// so the simulation is only run for small launches.
// Tiles of a launch with this pairing.
__host__ __device__ __forceinline__ int forward_tiles(int BH, int nqb, int pairing) {
  return BH * (pairing >= 2 ? nqb : (nqb + 1) >> 1);
}

// Pairing of a launch: single query blocks when there are fewer pairs than SMs (and the
// pattern allows it), else adjacent pairs or, under the causal mask, balanced ones when
// their snake schedule is lighter (choose_balanced_pairing).
int choose_balanced_pairing(int BH, int Nq, int Nk, int grid);
inline int choose_pairing(int BH, int Nq, int Nk, bool causal, bool allow_single, bool allow_balanced,
                          int num_sms, int* grid) {
  const int nqb = (Nq + kTileRows - 1) / kTileRows;
  const int pairs = forward_tiles(BH, nqb, 0);
  int pairing = 0;
  if (allow_single && nqb > 1 && pairs < num_sms) {
    pairing = 2;
  } else if (causal && allow_balanced) {
    const int g = pairs < num_sms ? pairs : num_sms;
    pairing = choose_balanced_pairing(BH, Nq, Nk, g);
  }
  const int tiles = forward_tiles(BH, nqb, pairing);
  *grid = tiles < num_sms ? tiles : num_sms;
  return pairing;
}

int choose_balanced_pairing(int BH, int Nq, int Nk, int grid) {
  const int nqb = (Nq + kTileRows - 1) / kTileRows;
  const int npairs = (nqb + 1) / 2;
  const long long ntiles = (long long)BH * npairs;
  if (ntiles > 8LL * grid) return 0;
  long long worst[2] = {0, 0};
  std::vector<long long> load(grid);
  for (int mode = 0; mode < 2; ++mode) {
    std::fill(load.begin(), load.end(), 0);
    for (long long t = 0; t < ntiles; ++t) {
      const long long r = t / BH;
      int qb0, qb1;
      if (mode) {
        qb0 = (int)r;
        qb1 = nqb - 1 - (int)r;
      } else {
        qb0 = 2 * (npairs - 1 - (int)r);
        qb1 = qb0 + 1;
      }
      const long long cost = visible_kv_blocks(qb0, Nq, Nk, true) +
                             ((qb1 < nqb && qb1 != qb0) ? visible_kv_blocks(qb1, Nq, Nk, true) : 0);
      const long long round = t / grid, pos = t % grid;
      load[(round & 1) ? grid - 1 - pos : pos] += cost;
    }
    worst[mode] = *std::max_element(load.begin(), load.end());
  }
  return worst[1] < worst[0] ? 1 : 0;
}

}  // namespace
}  // namespace fa
