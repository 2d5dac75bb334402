// sched.cuh -- tile order of the persistent tile kernels.
#pragma once

namespace fp8g {

// Grouped rasterisation: tiles are visited in groups of `group_m` consecutive
// M blocks, walking N within a group, so the CTAs resident at one time share
// few x row-blocks and few w column-blocks and re-read them from L2 (the
// grouped tile order of the "Kimi K3 (256k)" page, SM90 WGMMA paragraph).
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
  const int per_group = group_m * num_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// Work of one persistent worker (a CTA pair) out of `workers`.
//
// Without a split tail, worker r takes tiles r, r + workers, r + 2 workers,
// ... whole.  With it, only the first floor(tiles / workers) waves are taken
// whole; the K blocks of the remaining tiles, concatenated in tile order, are
// divided evenly between the first `tail_workers` workers, each taking one
// contiguous range, so that the last wave ends after a fraction of a tile
// instead of some workers running one tile longer than the rest.  A range
// cut at tile boundaries gives segments.  The segment holding a tile's first
// K block owns the tile: it adds the partial sums of that tile's other
// segments and writes y.  Any other segment is the first segment of its
// worker's range (later segments start on a tile boundary), so each worker
// publishes at most one partial sum, kept in slot `worker`.  The owner ends
// its range with its segment of the tile, which the workers after it start
// theirs with, so it rarely waits.  The host makes every tail range at least
// one K block long.
struct WorkUnit {
  int tile;    // tile index in raster order
  int k0, k1;  // K blocks [k0, k1) of the tile
  bool owner;  // true: write y (after adding the partials of workers owner+1 .. q_end-1)
  int q_end;
};

struct WorkIter {
  int me, workers, tail_workers, num_kb, n_full, tail_base, tail_tiles;
  int u;
  long long it, te;

  // tail_workers == 0: no split tail.
  __device__ WorkIter(int me_, int workers_, int num_tiles, int num_kb_, int tail_workers_)
      : me(me_), workers(workers_), tail_workers(tail_workers_), num_kb(num_kb_), u(0) {
    if (tail_workers > 0) {
      n_full = num_tiles / workers;
      tail_base = n_full * workers;
      tail_tiles = num_tiles - tail_base;
    } else {
      n_full = me < num_tiles ? (num_tiles - 1 - me) / workers + 1 : 0;
      tail_base = num_tiles;
      tail_tiles = 0;
    }
    it = tail_begin(me);
    te = tail_begin(me + 1);
  }

  // First K block (in the concatenated tail) of worker q's range.
  __device__ long long tail_begin(int q) const {
    if (tail_workers <= 0) return 0;
    if (q >= tail_workers) return static_cast<long long>(tail_tiles) * num_kb;
    return static_cast<long long>(tail_tiles) * num_kb * q / tail_workers;
  }

  __device__ bool next(WorkUnit& w) {
    if (u < n_full) {
      w.tile = me + u * workers;
      w.k0 = 0;
      w.k1 = num_kb;
      w.owner = true;
      w.q_end = me + 1;
      ++u;
      return true;
    }
    if (it >= te) return false;
    const int j = static_cast<int>(it / num_kb);
    const long long tile_first = static_cast<long long>(j) * num_kb;
    const long long tile_end = tile_first + num_kb;
    const long long seg_end = te < tile_end ? te : tile_end;
    w.tile = tail_base + j;
    w.k0 = static_cast<int>(it - tile_first);
    w.k1 = static_cast<int>(seg_end - tile_first);
    w.owner = (w.k0 == 0);
    int q = me + 1;
    if (w.owner)
      while (q < tail_workers && tail_begin(q) < tile_end) ++q;
    w.q_end = q;
    it = seg_end;
    return true;
  }
};

// Where a tile of the work list lies in x, w, y and scale.
struct TileGeom {
  int row;      // first x / y row of the 256-row tile
  int row_end;  // rows >= row_end belong to another group (or lie past M)
  int wrow;     // first w row of the tile
  int nb;       // N block: columns [nb BN, nb BN + BN)
  int sbase;    // offset of the tile's scales in the scale array
};

// Tile geometry of a (possibly grouped) layer, for tile indices visited in
// increasing order.  Without groups, tile t is (mb, nb) of the grouped
// raster over M x N.  With groups, group g owns rows [lo_g, hi_g) with
// lo_g = max(clamp(offs[g]), hi_{g-1}) and hi_g = max(clamp(offs[g+1]), lo_g)
// (clamp to [0, M]; hi_{-1} = 0), so groups never overlap whatever the
// offsets hold; it owns ceil((hi_g - lo_g) / 256) x nnb tiles, numbered after
// those of groups < g and rastered within the group.  The cursor walks the
// group offsets forward once.
struct TileMapper {
  const int* offs;  // nullptr: one group
  int groups, M, N, bn, nnb, num_m_blk, group_m;
  int g, lo, hi, m_blocks;
  long long before;  // tiles of groups < g

  __device__ TileMapper(const int* offs_, int groups_, int M_, int N_, int bn_, int nnb_,
                        int num_m_blk_, int group_m_)
      : offs(offs_), groups(groups_), M(M_), N(N_), bn(bn_), nnb(nnb_), num_m_blk(num_m_blk_),
        group_m(group_m_), g(0), lo(0), hi(0), m_blocks(0), before(0) {
    if (offs) load(0, 0);
  }

  __device__ int clamp_row(int v) const { return v < 0 ? 0 : (v > M ? M : v); }

  // Group gg's rows, given the end of group gg - 1's rows.
  __device__ void load(int gg, int prev_hi) {
    g = gg;
    if (gg >= groups) {
      lo = hi = M;
      m_blocks = 0;
      return;
    }
    const int l = clamp_row(__ldg(offs + gg));
    lo = l < prev_hi ? prev_hi : l;
    const int h = clamp_row(__ldg(offs + gg + 1));
    hi = h < lo ? lo : h;
    m_blocks = (hi - lo + 255) / 256;
  }

  // Tiles of the whole layer.
  __device__ long long total() const {
    if (!offs) return static_cast<long long>(num_m_blk) * nnb;
    long long t = 0;
    int prev_hi = 0;
    for (int gg = 0; gg < groups; ++gg) {
      int l = clamp_row(__ldg(offs + gg));
      if (l < prev_hi) l = prev_hi;
      int h = clamp_row(__ldg(offs + gg + 1));
      if (h < l) h = l;
      t += static_cast<long long>((h - l + 255) / 256) * nnb;
      prev_hi = h;
    }
    return t;
  }

  __device__ TileGeom at(int t) {
    TileGeom r;
    int mb, nb;
    if (!offs) {
      tile_coords(t, num_m_blk, nnb, group_m, mb, nb);
      r.row = mb * 256;
      r.row_end = M;
      r.wrow = nb * bn;
      r.nb = nb;
      r.sbase = 0;
      return r;
    }
    while (g < groups && t >= before + static_cast<long long>(m_blocks) * nnb) {
      before += static_cast<long long>(m_blocks) * nnb;
      load(g + 1, hi);
    }
    tile_coords(static_cast<int>(t - before), m_blocks > 0 ? m_blocks : 1, nnb, group_m, mb, nb);
    r.row = lo + mb * 256;
    r.row_end = hi;
    r.wrow = g * N + nb * bn;
    r.nb = nb;
    r.sbase = g * N;
    return r;
  }
};

}  // namespace fp8g
