// Checks of the host/device-shared scheduling logic of lin_internal.h, run on
// the CPU by tests/test_host_logic.py: the clustered kernels' tile order and
// the split plan of their persistent launches. Prints "ok" or the first
// violated property.
#include <cstdio>
#include <vector>

#include "lin_internal.h"

static int fail(const char* what, int a, int b, int c, int d) {
  std::printf("FAIL %s (%d %d %d %d)\n", what, a, b, c, d);
  return 1;
}

int main() {
  // tile_coords: a bijection of [0, num_m * num_ng) onto the grid; one band
  // (band <= 0 or >= num_ng) is the row-major order; with bands, tiles of
  // band b come before those of band b + 1 and the column group varies
  // fastest inside a band.
  const int ms[] = {1, 3, 4, 7, 128};
  const int ngs[] = {1, 2, 5, 16, 17};
  const int bands[] = {0, 1, 2, 3, 4, 8, 16, 100};
  for (int num_m : ms)
    for (int num_ng : ngs)
      for (int band : bands) {
        const int n = num_m * num_ng;
        std::vector<int> seen(n, 0);
        int prev_b = 0;
        for (int t = 0; t < n; ++t) {
          const lin::TileRC rc = lin::tile_coords(t, num_m, num_ng, band);
          if (rc.m < 0 || rc.m >= num_m || rc.ng < 0 || rc.ng >= num_ng)
            return fail("tile out of the grid", num_m, num_ng, band, t);
          if (seen[rc.m * num_ng + rc.ng]++) return fail("tile visited twice", num_m, num_ng, band, t);
          if (band <= 0 || band >= num_ng) {
            if (rc.m != t / num_ng || rc.ng != t % num_ng)
              return fail("one band is not row-major", num_m, num_ng, band, t);
            continue;
          }
          const int b = rc.ng / band;
          if (b < prev_b) return fail("bands out of order", num_m, num_ng, band, t);
          prev_b = b;
          if (t > 0) {   // within a band, the column group varies fastest
            const lin::TileRC p = lin::tile_coords(t - 1, num_m, num_ng, band);
            if (p.ng / band == b && p.m == rc.m && p.ng + 1 != rc.ng)
              return fail("column group not fastest", num_m, num_ng, band, t);
            if (p.ng / band == b && p.m != rc.m && (p.m + 1 != rc.m || rc.ng != b * band))
              return fail("row step inside a band", num_m, num_ng, band, t);
          }
        }
      }

  // split_plan: r whole rounds on every cluster plus rem tail tiles, each
  // cut into s >= 2 K ranges of at least kSplitMinKb k-blocks that fit the
  // clusters; no split when the rounds are whole or a range would be short.
  for (int tiles = 1; tiles <= 300; tiles += 7)
    for (int clusters = 1; clusters <= 152; clusters += 5)
      for (int nkb = 1; nkb <= 256; nkb *= 2) {
        const lin::SplitPlan p = lin::split_plan(tiles, clusters, nkb);
        if (p.s < 2) {
          if (p.s != 1) return fail("no split must have s == 1", tiles, clusters, nkb, p.s);
          continue;
        }
        if (p.r * clusters + p.rem != tiles) return fail("tiles not covered", tiles, clusters, nkb, p.s);
        if (p.rem <= 0 || p.rem >= clusters) return fail("tail not partial", tiles, clusters, nkb, p.s);
        if (p.rem * p.s > clusters) return fail("tail ranges exceed clusters", tiles, clusters, nkb, p.s);
        if (p.s * lin::kSplitMinKb > nkb) return fail("K range too short", tiles, clusters, nkb, p.s);
        if (tiles % clusters == 0) return fail("split with whole rounds", tiles, clusters, nkb, p.s);
      }
  std::printf("ok\n");
  return 0;
}
