// Work items of the query-tile-parallel kernels (the forward and the
// backward's Dvec pass), head-paired where that helps.
#pragma once

#include "attn_common.cuh"

namespace attn {

// The two 128-row query tiles of one work item: tile t holds rows qs[t].. of
// query head hq[t] (both heads in kv group g of batch b) and needs K/V tiles
// [j_lo[t], n_kv[t]). Unpaired, the tiles are consecutive row blocks of one
// head (FwdItem). Head-paired (causal masking with an even number of query
// heads per kv head), they are the same rows of two heads of one group: both
// need the same K/V tiles, so every K/V step feeds both tiles, where the
// consecutive tiles' key ranges are one tile apart (with a 128-key window a
// step of tile A alone, one of both and one of tile B alone).
struct TileItem {
  int b, g;
  int hq[2], qs[2];
  int n_kv[2], j_lo[2];
};

template <class P>
__host__ __device__ __forceinline__ int tile_n_items(const P& p, bool pair) {
  return pair ? p.B * (p.Hq / 2) * ((p.S + 127) / 128) : p.B * p.Hq * p.n_qblocks;
}

// Item i, longest first: paired items take head pair i % (B Hq / 2) of query
// tile n_qt - 1 - i / (B Hq / 2). P is a parameter block with B, Hq, G, S,
// causal, window and n_qblocks.
template <bool WIN, class P>
__device__ __forceinline__ TileItem tile_item(const P& p, bool pair, int i) {
  constexpr int BT = 128;  // rows of a query tile, keys of a K/V tile
  TileItem it;
  if (!pair) {
    const FwdItem f = fwd_item<WIN>(p, i);
    it.b = f.b;
    it.g = f.g;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      it.hq[t] = f.hq;
      it.qs[t] = f.q0 + t * BT;
      it.n_kv[t] = f.n_kv[t];
      it.j_lo[t] = f.j_lo[t];
    }
    return it;
  }
  const int hp = p.Hq / 2, bhp = p.B * hp;
  const int nt = (p.S + BT - 1) / BT;
  const int bh = i % bhp;
  const int h0 = 2 * (bh % hp);
  const int qs = (nt - 1 - i / bhp) * BT;
  const int n_kv = p.causal ? min(qs / BT + 1, nt) : nt;
  const int j_lo = WIN ? min(max(0, qs - p.window + 1) / BT, n_kv - 1) : 0;
  it.b = bh / hp;
  it.g = h0 / p.G;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.hq[t] = h0 + t;
    it.qs[t] = qs;
    it.n_kv[t] = n_kv;
    it.j_lo[t] = j_lo;
  }
  return it;
}

// Head pairing: with causal masking and an even number of query heads per kv
// head.
template <class P>
inline bool tile_pair_heads(const P& p) {
  return p.causal && p.G % 2 == 0;
}

}  // namespace attn
