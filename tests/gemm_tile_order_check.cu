// Host-side check of the GEMM's tile order (make_tile_order / tile_of in
// gemm_fp4.cu): for every shape of a sweep, the indices 0 .. ntiles-1 map
// onto the MT x NT output tiles one to one; with the balanced order each
// round j (indices jU .. jU + U - 1) covers the same tiles as plain row
// order, and no order gives a CTA pair more MMA work than plain row order
// (a half-width tile counts half).  Exit status 0 when all hold.
#include "gemm_fp4.cu"

#include <cstdio>
#include <vector>

using sixbit::TileOrder;
using sixbit::make_tile_order;
using sixbit::tile_of;

namespace {

// largest per-pair work in half-tile units (full tile 2, half tile 1)
int makespan(const TileOrder& o, bool plain) {
  std::vector<int> w(o.U, 0);
  for (int i = 0; i < o.ntiles; ++i) {
    int mt = i / o.NT, nt = i % o.NT;
    if (!plain) tile_of(o, i, mt, nt);
    w[i % o.U] += o.half && nt == o.NT - 1 ? 1 : 2;
  }
  int m = 0;
  for (int x : w) m = x > m ? x : m;
  return m;
}

bool check(int MT, int NT, int U, bool half) {
  const TileOrder o = make_tile_order(MT, NT, U, half);
  std::vector<char> seen(size_t(MT) * NT, 0);
  for (int i = 0; i < o.ntiles; ++i) {
    int mt = -1, nt = -1;
    tile_of(o, i, mt, nt);
    if (mt < 0 || mt >= MT || nt < 0 || nt >= NT || seen[size_t(mt) * NT + nt]++) {
      std::printf("not a bijection: MT=%d NT=%d U=%d half=%d index %d -> (%d, %d)\n", MT, NT, U, half, i, mt, nt);
      return false;
    }
    const int pos = mt * NT + nt, j = i / U;
    if (o.bal && (pos < j * U || pos >= (j + 1) * U)) {
      std::printf("round changed: MT=%d NT=%d U=%d index %d -> row-order position %d\n", MT, NT, U, i, pos);
      return false;
    }
  }
  const int mk = makespan(o, false), mk0 = makespan(o, true);
  if (mk > mk0 || (o.bal && mk > 2 * (o.ntiles / U))) {
    std::printf("load: MT=%d NT=%d U=%d half=%d: %d half-tiles vs %d in row order\n", MT, NT, U, half, mk, mk0);
    return false;
  }
  return true;
}

}  // namespace

int main() {
  long shapes = 0, balanced = 0;
  for (int MT = 1; MT <= 120; ++MT)
    for (int NT = 1; NT <= 40; ++NT)
      for (int U = 1; U <= 76 && U <= MT * NT; ++U)
        for (int half = 0; half < 2; ++half) {
          if (!check(MT, NT, U, half != 0)) return 1;
          ++shapes;
          balanced += make_tile_order(MT, NT, U, half != 0).bal;
        }
  // the 2B-class layers on 76 pairs: N = 1920 (7.5 tiles) and N = 5760 (22.5)
  const int want[2][3] = {{70, 8, 14}, {70, 23, 42}};
  for (const auto& s : want) {
    const TileOrder o = make_tile_order(s[0], s[1], 76, true);
    if (!o.bal || makespan(o, false) != s[2]) {
      std::printf("2B shape MT=%d NT=%d: bal=%d, load %d half-tiles (want %d)\n", s[0], s[1], o.bal,
                  makespan(o, false), s[2]);
      return 1;
    }
  }
  std::printf("ok: %ld shapes, %ld with the balanced order\n", shapes, balanced);
  return 0;
}
