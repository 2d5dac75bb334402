// sched_check.cpp -- host build of the tile scheduler (sched.cuh) and checks
// of the properties the persistent tile kernels rely on, over many seeded
// parameter sets.  Prints "ok <cases>" and exits 0, or prints the first
// failures and exits 1.  Built and run by tests/test_sched_host.py.
#include <algorithm>
#include <cstdio>
#include <map>
#include <random>
#include <vector>

#define __device__
#define __forceinline__ inline
using std::min;
template <class T>
static inline T __ldg(const T* p) {
  return *p;
}
#include "sched.cuh"

using fp8g::TileGeom;
using fp8g::TileMapper;
using fp8g::WorkIter;
using fp8g::WorkUnit;

static long long g_fails = 0;
#define CHECK(cond, ...)                                              \
  do {                                                                \
    if (!(cond)) {                                                    \
      if (g_fails++ < 12) {                                           \
        std::fprintf(stderr, "FAIL line %d (%s): ", __LINE__, #cond); \
        std::fprintf(stderr, __VA_ARGS__);                            \
        std::fprintf(stderr, "\n");                                   \
      }                                                               \
    }                                                                 \
  } while (0)

// Grouped raster: a bijection of [0, num_m * num_n) onto the M x N blocks
// that visits group_m M blocks (fewer in the last group) before moving on.
static void check_raster(int num_m, int num_n, int group_m) {
  std::vector<int> seen(static_cast<size_t>(num_m) * num_n, 0);
  for (int t = 0; t < num_m * num_n; ++t) {
    int mb = -1, nb = -1;
    fp8g::tile_coords(t, num_m, num_n, group_m, mb, nb);
    CHECK(mb >= 0 && mb < num_m && nb >= 0 && nb < num_n, "t=%d -> (%d, %d) of %dx%d", t, mb,
          nb, num_m, num_n);
    if (mb < 0 || mb >= num_m || nb < 0 || nb >= num_n) continue;
    ++seen[static_cast<size_t>(mb) * num_n + nb];
    CHECK(mb / group_m == t / (group_m * num_n), "t=%d in group %d, mb=%d", t,
          t / (group_m * num_n), mb);
  }
  for (size_t i = 0; i < seen.size(); ++i)
    CHECK(seen[i] == 1, "block %zu visited %d times (%dx%d, group %d)", i, seen[i], num_m, num_n,
          group_m);
}

// The host's number of tail workers (as the library's planner chooses it): at
// most two per tail tile and at most the workers, every range at least one K
// block, and more workers than tail tiles (else no split).
static int host_tail_workers(long long tiles, int workers, int num_kb) {
  const long long rem = tiles % workers;
  if (rem == 0) return 0;
  long long tw = std::min<long long>(workers, rem * 2);
  tw = std::min<long long>(tw, rem * num_kb);
  return tw > rem ? static_cast<int>(tw) : 0;
}

static void check_work(int workers, int tiles, int num_kb, int tail_workers, bool host_rule) {
  std::vector<std::vector<WorkUnit>> per(workers);
  for (int me = 0; me < workers; ++me) {
    WorkIter wi(me, workers, tiles, num_kb, tail_workers);
    WorkUnit w;
    int guard = 0;
    while (wi.next(w) && guard++ < (1 << 20)) per[me].push_back(w);
  }
  const int n_full = tail_workers > 0 ? tiles / workers : 0;
  std::vector<int> cover(static_cast<size_t>(tiles) * num_kb, 0);
  std::vector<int> owners(tiles, 0);
  // non-owner segments by tile: (worker, k0, k1)
  std::map<int, std::vector<std::vector<int>>> parts;
  for (int me = 0; me < workers; ++me) {
    int non_owner = 0;
    for (size_t i = 0; i < per[me].size(); ++i) {
      const WorkUnit& u = per[me][i];
      CHECK(u.tile >= 0 && u.tile < tiles && u.k0 >= 0 && u.k0 < u.k1 && u.k1 <= num_kb,
            "worker %d unit %zu: tile %d [%d, %d)", me, i, u.tile, u.k0, u.k1);
      if (!(u.tile >= 0 && u.tile < tiles && u.k0 >= 0 && u.k0 < u.k1 && u.k1 <= num_kb))
        continue;
      for (int kb = u.k0; kb < u.k1; ++kb) ++cover[static_cast<size_t>(u.tile) * num_kb + kb];
      CHECK(u.owner == (u.k0 == 0), "worker %d tile %d: owner %d with k0 %d", me, u.tile,
            static_cast<int>(u.owner), u.k0);
      if (u.owner) {
        ++owners[u.tile];
      } else {
        ++non_owner;
        // a partial comes from the first unit of the worker's tail range
        CHECK(static_cast<int>(i) == n_full, "worker %d: partial at unit %zu, tail starts at %d",
              me, i, n_full);
        parts[u.tile].push_back({me, u.k0, u.k1});
      }
      if (tail_workers == 0) {
        CHECK(u.tile == me + static_cast<int>(i) * workers && u.k0 == 0 && u.k1 == num_kb &&
                  u.q_end == me + 1,
              "worker %d unit %zu: tile %d [%d, %d) q_end %d without a split tail", me, i,
              u.tile, u.k0, u.k1, u.q_end);
      } else if (static_cast<int>(i) < n_full) {
        CHECK(u.tile == me + static_cast<int>(i) * workers && u.k0 == 0 && u.k1 == num_kb,
              "worker %d whole unit %zu: tile %d", me, i, u.tile);
      }
    }
    CHECK(non_owner <= 1, "worker %d publishes %d partial sums", me, non_owner);
    if (tail_workers > 0 && me < tail_workers)
      CHECK(static_cast<int>(per[me].size()) > n_full, "tail worker %d has an empty range", me);
  }
  for (size_t i = 0; i < cover.size(); ++i)
    CHECK(cover[i] == 1, "tile %zu K block %zu covered %d times (workers %d, tiles %d, kb %d, tw %d)",
          i / num_kb, i % num_kb, cover[i], workers, tiles, num_kb, tail_workers);
  for (int t = 0; t < tiles; ++t) CHECK(owners[t] == 1, "tile %d has %d owners", t, owners[t]);
  // an owner adds the partials of workers owner+1 .. q_end-1, which hold the
  // rest of its tile in order; a split tile is its owner's last unit
  for (int me = 0; me < workers; ++me) {
    for (size_t i = 0; i < per[me].size(); ++i) {
      const WorkUnit& u = per[me][i];
      if (!u.owner) continue;
      const auto it = parts.find(u.tile);
      const std::vector<std::vector<int>> none;
      const std::vector<std::vector<int>>& ps = it == parts.end() ? none : it->second;
      CHECK(u.q_end - (me + 1) == static_cast<int>(ps.size()),
            "tile %d: q_end %d for owner %d but %zu contributors", u.tile, u.q_end, me, ps.size());
      int k = u.k1;
      for (size_t j = 0; j < ps.size(); ++j) {
        CHECK(ps[j][0] == me + 1 + static_cast<int>(j), "tile %d: contributor %zu is worker %d",
              u.tile, j, ps[j][0]);
        CHECK(ps[j][1] == k, "tile %d: contributor %zu starts at %d, expected %d", u.tile, j,
              ps[j][1], k);
        k = ps[j][2];
      }
      CHECK(k == num_kb, "tile %d: segments end at %d of %d", u.tile, k, num_kb);
      if (!ps.empty())
        CHECK(i + 1 == per[me].size(), "tile %d split but not the last unit of owner %d", u.tile,
              me);
      // with at most two tail workers per tail tile every range holds at
      // least half a tile (rounded down), so a tile meets at most three
      if (host_rule)
        CHECK(static_cast<int>(ps.size()) + 1 <= 3, "tile %d in %zu segments", u.tile,
              ps.size() + 1);
      if (tail_workers > 0 && ps.size() + 1 > 1) {
        const long long tail_kb = static_cast<long long>(tiles % workers) * num_kb;
        const long long lmin = tail_kb / tail_workers;  // shortest range
        CHECK(lmin >= 1 && static_cast<long long>(ps.size()) <= (num_kb - 1 + lmin - 1) / lmin,
              "tile %d in %zu segments, ranges of %lld K blocks or more", u.tile, ps.size() + 1,
              lmin);
      }
    }
  }
}

// Tiles of a grouped layer: group g owns rows [lo_g, hi_g) (offsets clamped
// to [0, M], each group starting no earlier than the previous one ends), cut
// into 256-row blocks; every (row block, N block) of every group is visited
// once, in increasing tile order.
static void check_groups(const std::vector<int>& offs, int M, int N, int bn, int group_m) {
  const int groups = static_cast<int>(offs.size()) - 1;
  const int nnb = (N + bn - 1) / bn;
  std::vector<int> lo(groups), hi(groups);
  int prev = 0;
  long long expect = 0;
  for (int g = 0; g < groups; ++g) {
    const int l = std::min(std::max(offs[g], 0), M);
    const int h = std::min(std::max(offs[g + 1], 0), M);
    lo[g] = std::max(l, prev);
    hi[g] = std::max(h, lo[g]);
    prev = hi[g];
    expect += static_cast<long long>((hi[g] - lo[g] + 255) / 256) * nnb;
  }
  TileMapper tm(offs.data(), groups, M, N, bn, nnb, (M + 255) / 256, group_m);
  const long long total = tm.total();
  CHECK(total == expect, "total %lld, expected %lld", total, expect);
  std::map<long long, int> seen;
  for (long long t = 0; t < total; ++t) {
    const TileGeom tg = tm.at(static_cast<int>(t));
    const int g = N > 0 ? tg.sbase / N : 0;
    CHECK(g >= 0 && g < groups && tg.sbase == g * N, "tile %lld: scale base %d", t, tg.sbase);
    if (g < 0 || g >= groups) continue;
    CHECK(tg.row >= lo[g] && tg.row < hi[g] && (tg.row - lo[g]) % 256 == 0 && tg.row_end == hi[g],
          "tile %lld: rows %d.. of group %d [%d, %d), end %d", t, tg.row, g, lo[g], hi[g],
          tg.row_end);
    CHECK(tg.nb >= 0 && tg.nb < nnb && tg.wrow == g * N + tg.nb * bn,
          "tile %lld: nb %d, w row %d", t, tg.nb, tg.wrow);
    const long long key = (static_cast<long long>(g) * (M / 256 + 2) + (tg.row - lo[g]) / 256) *
                              nnb + tg.nb;
    ++seen[key];
  }
  CHECK(static_cast<long long>(seen.size()) == expect, "%zu distinct tiles of %lld", seen.size(),
        expect);
  for (const auto& kv : seen) CHECK(kv.second == 1, "tile key %lld visited %d times", kv.first, kv.second);
}

// Without group offsets the mapper is the plain raster.
static void check_plain_mapper(int M, int N, int bn, int group_m) {
  const int nnb = (N + bn - 1) / bn;
  const int nm = (M + 255) / 256;
  TileMapper tm(nullptr, 0, M, N, bn, nnb, nm, group_m);
  CHECK(tm.total() == static_cast<long long>(nm) * nnb, "plain total");
  for (int t = 0; t < nm * nnb; ++t) {
    int mb, nb;
    fp8g::tile_coords(t, nm, nnb, group_m, mb, nb);
    const TileGeom tg = tm.at(t);
    CHECK(tg.row == mb * 256 && tg.row_end == M && tg.nb == nb && tg.wrow == nb * bn &&
              tg.sbase == 0,
          "plain tile %d", t);
  }
}

int main() {
  std::mt19937 rng(20240607u);
  auto uni = [&](int a, int b) { return std::uniform_int_distribution<int>(a, b)(rng); };
  long long cases = 0;
  for (int i = 0; i < 400; ++i, ++cases) check_raster(uni(1, 40), uni(1, 40), uni(1, 20));
  check_raster(16, 19, 16);  // the 4096^3 workload with 256 x 224 tiles
  ++cases;
  // whole tiles, and every split-tail worker count the kernels accept
  std::vector<std::vector<int>> fixed = {{76, 304, 32}, {76, 152, 33}, {76, 1792, 32},
                                         {76, 19, 32},  {76, 77, 1},   {76, 75, 3},
                                         {1, 5, 7},     {3, 0, 4},     {76, 100, 2}};
  for (int i = 0; i < 1500; ++i) {
    std::vector<int> p = i < static_cast<int>(fixed.size())
                             ? fixed[i]
                             : std::vector<int>{uni(1, 80), uni(0, 400), uni(1, 40)};
    const int workers = p[0], tiles = p[1], num_kb = p[2];
    check_work(workers, tiles, num_kb, 0, true);
    ++cases;
    const int rem = tiles % workers;
    const int host = host_tail_workers(tiles, workers, num_kb);
    if (host > 0) {
      check_work(workers, tiles, num_kb, host, true);
      ++cases;
    }
    if (rem > 0) {
      const int hi = std::min<long long>(workers, static_cast<long long>(rem) * num_kb);
      for (int tw = rem + 1; tw <= hi; tw += std::max(1, (hi - rem) / 4)) {
        check_work(workers, tiles, num_kb, tw, false);
        ++cases;
      }
    }
  }
  for (int i = 0; i < 600; ++i, ++cases) {
    const int groups = uni(1, 12);
    const int M = uni(0, 3000);
    std::vector<int> offs(groups + 1);
    const bool sorted = uni(0, 2) != 0;
    for (int g = 0; g <= groups; ++g) offs[g] = uni(-100, M + 100);
    if (sorted) std::sort(offs.begin(), offs.end());
    const int bn = 32 * uni(2, 8);
    check_groups(offs, M, uni(1, 1000), bn, uni(1, 16));
  }
  check_groups({0, 45, 45, 301, 333, 700, 1000}, 1000, 640, 256, 16);
  check_groups({40, 100, 50, 2000, 20}, 300, 384, 128, 16);
  for (int i = 0; i < 200; ++i, ++cases) check_plain_mapper(uni(1, 5000), uni(1, 5000), 32 * uni(2, 8), uni(1, 16));
  if (g_fails) {
    std::printf("%lld failures in %lld cases\n", g_fails, cases);
    return 1;
  }
  std::printf("ok %lld cases\n", cases);
  return 0;
}
