// Host check of the tree-verify attention's work division (attn_plan.cuh):
// for random batches and grid sizes, every CTA walks its items and the union
// must cover every KV tile of every (request, KV head, M-tile pair) group
// exactly once, in order, with consistent split counts and partial slots.
// Prints "OK <cases>" or the first violation; exit status 0 only on OK.
//
// The per-request cost below restates the kernel's planner: T KV tiles of 128
// keys, MT M tiles of 128 rows, MP = ceil(MT / 2) pairs, a tile of a pair with
// nt active M tiles costing nt + 1 + tx, eh more units at the start of a group and
// ee more at its end (a few for the kernels; drawn at random here); CTAs that
// receive work: max(1, min(grid, W / (3 + tx))).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <set>
#include <tuple>
#include <vector>

#include "attn_plan.cuh"

using namespace tv::attn;

struct Rec {
  int cta, tile_begin, tile_end, k0, n_splits, slot0, my_slot, nt;
};

static int fail(const char* what, int c, int b, int g, int mp) {
  std::printf("FAIL case %d: %s (request %d, head %d, pair %d)\n", c, what, b, g, mp);
  return 1;
}

int main(int argc, char** argv) {
  const int n_cases = argc > 1 ? std::atoi(argv[1]) : 400;
  std::mt19937_64 rng(12345);
  auto uni = [&](int lo, int hi) { return (int)std::uniform_int_distribution<int>(lo, hi)(rng); };
  const int grids[] = {1, 2, 7, 148, 152, 304};
  const int heads[] = {1, 2, 4, 8, 32};
  const int groups[] = {1, 2, 4, 8, 16, 32, 64};
  for (int c = 0; c < n_cases; ++c) {
    const int B = uni(1, c % 5 == 0 ? 300 : 40);
    const int Hkv = heads[uni(0, 4)];
    const int G = groups[uni(0, 6)];
    const int grid = grids[uni(0, 5)];
    const int maxL = (c % 3 == 0) ? 40000 : 3000;
    // the charges the kernels use (one CTA: 6 at each end, low-bit tiles 2 more;
    // CTA pairs: 8) among others
    const int ehs[] = {0, 1, 3, 6, 8, 40};
    const int eh = ehs[uni(0, 5)], ee = ehs[uni(0, 5)];
    const int txs[] = {0, 0, 1, 2, 4, 9};
    const int tx = txs[uni(0, 5)];
    std::vector<int64_t> start(B + 1);
    std::vector<int32_t> T(B), MT(B);
    int64_t W = 0;
    for (int b = 0; b < B; ++b) {
      const bool skipped = uni(0, 9) == 0;
      const int N = uni(1, 64), L = uni(0, maxL);
      T[b] = skipped ? 0 : (L + N + 127) / 128;
      MT[b] = skipped ? 0 : (N * G + 127) / 128;
      start[b] = W;
      if (T[b] > 0)
        W += (int64_t)Hkv * ((int64_t)T[b] * (MT[b] + (int64_t)(1 + tx) * ((MT[b] + 1) / 2)) +
                             (int64_t)(eh + ee) * ((MT[b] + 1) / 2));
    }
    start[B] = W;
    if (W == 0) continue;
    PlanView pv;
    pv.start = start.data();
    pv.T = T.data();
    pv.MT = MT.data();
    pv.B = B;
    pv.Hkv = Hkv;
    pv.eh = eh;
    pv.ee = ee;
    pv.tx = tx;
    pv.W = W;
    pv.C = (int)std::max<int64_t>(1, std::min<int64_t>(grid, W / (3 + tx)));
    pv.narrow = (int64_t)(pv.C + 1) * W < (int64_t(1) << 32);

    std::map<std::tuple<int, int, int>, std::vector<Rec>> by_group;
    for (int cta = 0; cta < pv.C; ++cta) {
      ItemIter it;
      iter_init(it, pv, cta);
      Item item;
      int items = 0;
      while (iter_next(it, pv, cta, item)) {
        if (++items > 100000) return fail("runaway iterator", c, -1, -1, -1);
        by_group[{item.b, item.g, item.mp}].push_back(
            {cta, item.tile_begin, item.tile_end, item.k0, item.n_splits, item.slot0, item.my_slot, item.nt});
      }
    }
    // every group of every request with work: tiles covered once, in CTA order
    std::map<int, std::tuple<int, int, int>> slot_owner;  // slot -> group, for groups with splits
    for (int b = 0; b < B; ++b) {
      if (T[b] == 0) continue;
      const int MP = (MT[b] + 1) / 2;
      for (int g = 0; g < Hkv; ++g)
        for (int mp = 0; mp < MP; ++mp) {
          auto f = by_group.find({b, g, mp});
          if (f == by_group.end()) return fail("group never planned", c, b, g, mp);
          const std::vector<Rec>& rs = f->second;
          const int ns = (int)rs.size();
          int next_tile = 0;
          for (int s = 0; s < ns; ++s) {
            const Rec& r = rs[s];
            if (r.tile_begin != next_tile || r.tile_end <= r.tile_begin) return fail("tiles not contiguous", c, b, g, mp);
            next_tile = r.tile_end;
            if (r.n_splits != ns) return fail("split count differs from the CTAs holding the group", c, b, g, mp);
            if (r.k0 != rs[0].cta || r.cta != rs[0].cta + s) return fail("splits not on consecutive CTAs", c, b, g, mp);
            if (r.nt != imin32(2, MT[b] - 2 * mp)) return fail("active M tiles", c, b, g, mp);
            Item view;
            view.k0 = r.k0;
            view.slot0 = r.slot0;
            if (ns > 1 && r.my_slot != split_slot(view, s)) return fail("split writes a slot the merge does not read", c, b, g, mp);
            if (ns > 1) {
              auto o = slot_owner.find(r.my_slot);
              if (o != slot_owner.end() && o->second != std::make_tuple(b, g, mp))
                return fail("two split groups share a partial slot", c, b, g, mp);
              slot_owner[r.my_slot] = {b, g, mp};
              if (r.my_slot < 2 * r.cta || r.my_slot > 2 * r.cta + 1) return fail("slot outside the CTA's pair", c, b, g, mp);
            }
          }
          if (next_tile != T[b]) return fail("tiles missing at the end", c, b, g, mp);
          by_group.erase(f);
        }
    }
    if (!by_group.empty()) {
      auto k = by_group.begin()->first;
      return fail("item for a group without work", c, std::get<0>(k), std::get<1>(k), std::get<2>(k));
    }
  }
  std::printf("OK %d\n", n_cases);
  return 0;
}
