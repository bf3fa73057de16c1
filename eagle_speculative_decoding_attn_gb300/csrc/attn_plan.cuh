// Work division of the tree-verify attention kernel.  Every role of a CTA
// computes the same plan and walks the same items with these functions; they
// are plain integer arithmetic, compiled for the device by the kernel and for
// the host by the plan's tests.
//
// A work group is (request, KV head, M-tile pair); a KV tile of a group with nt
// active M tiles costs nt + 1 + tx units (tx: a per-tile cost that does not grow
// with nt, such as decoding a low-bit cache; 0 charges none), the start of a
// group eh more and its end ee more (the fixed costs of an item: the pipeline's
// restart, the epilogue and a split's merge; 0 charges none), and CTA k takes the contiguous cost range
// [cut(k), cut(k + 1)) of the whole batch.  At most W / (3 + tx) CTAs take work,
// so each range holds the first unit of at least one tile.  A group cut between CTAs is split: each split writes a partial into
// its slot and the last to arrive merges.
#ifndef TV_ATTN_PLAN_CUH_
#define TV_ATTN_PLAN_CUH_

#include <cstdint>

#ifdef __CUDACC__
#define TV_PLAN_INL __host__ __device__ __forceinline__
#define TV_PLAN_FN __host__ __device__ inline
#else
#define TV_PLAN_INL inline
#define TV_PLAN_FN inline
#endif

namespace tv {
namespace attn {

TV_PLAN_INL int imin32(int a, int b) { return a < b ? a : b; }
TV_PLAN_INL uint32_t umin32(uint32_t a, uint32_t b) { return a < b ? a : b; }
TV_PLAN_INL int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
TV_PLAN_INL int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }
// ceil(a / c) for a cost per tile c >= 2, 0 when a <= 0 (no division for c = 2)
TV_PLAN_INL int64_t ceil_div_c(int64_t a, int c) {
  if (a <= 0) return 0;
  if (c == 2) return (a + 1) >> 1;
  if (c == 3) return (a + 2) / 3;
  return (a + c - 1) / c;
}

struct PlanView {
  const int64_t* start;  // cost position of each request's first group; start[B] = W
  const int32_t* T;      // KV tiles of each request (0 = request skipped)
  const int32_t* MT;     // M tiles of each request
  int B, Hkv;
  int eh, ee;            // cost units at the start and at the end of a group (0: none)
  int tx;                // cost units of a KV tile on top of nt + 1 (0: none)
  int64_t W;             // total cost (< 2^40, so k * W fits in 64 bits)
  int C;                 // CTAs that receive work
  bool narrow;           // (C + 1) * W < 2^32: 32-bit division suffices
  // first cost position of CTA k, and the CTA owning cost position x
  TV_PLAN_INL int64_t cut(int k) const {
    if (narrow) return ((uint32_t)k * (uint32_t)W + (uint32_t)(C - 1)) / (uint32_t)C;
    return ((int64_t)k * W + C - 1) / C;
  }
  TV_PLAN_INL int owner(int64_t x) const {
    if (narrow) return (int)umin32((uint32_t)(C - 1), ((uint32_t)x * (uint32_t)C) / (uint32_t)W);
    return (int)imin64(C - 1, x * C / W);
  }
};

struct Item {
  int b, g, mp, nt;           // request, KV head, M-tile pair, active M tiles
  int tile_begin, tile_end;   // KV tiles of this item
  int k0, n_splits;           // first CTA of the group, number of splits
  int slot0;                  // partial slot of split 0
  int my_slot;                // partial slot of this CTA's split
};

// Iterates this CTA's items in the global (request, KV head, pair, tile) order.
// A tile belongs to the CTA whose cost range holds the tile's first cost unit;
// a tile of a group with nt active M tiles costs nt + 1 + tx units, and the group's
// tiles start eh units after the group (its end carries ee more).
struct ItemIter {
  int b, j;           // request and group index within it (j = g * MP + mp)
  int64_t gstart;     // cost position of the current group (its first tile starts eh later)
  int c_prev;         // cost per tile of the group before the current one (0: none)
  int produced;
  int64_t lo, hi;     // this CTA's cost range
};

TV_PLAN_FN void iter_init(ItemIter& it, const PlanView& pv, int cta) {
  it.produced = 0;
  it.lo = pv.cut(cta);
  it.hi = pv.cut(cta + 1);
  it.c_prev = 0;
  // largest b with start[b] <= lo (it has a non-zero cost), then its group
  int lo_b = 0, hi_b = pv.B;
  while (hi_b - lo_b > 1) {
    const int mid = (lo_b + hi_b) >> 1;
    if (pv.start[mid] <= it.lo) lo_b = mid; else hi_b = mid;
  }
  int b = lo_b;
  while (b < pv.B && pv.T[b] == 0) ++b;
  it.b = b;
  it.j = 0;
  it.gstart = b < pv.B ? pv.start[b] : pv.W;
  if (b < pv.B) {
    const int T = pv.T[b], MT = pv.MT[b], MP = (MT + 1) / 2;
    const int64_t per_g = (int64_t)T * (MT + (int64_t)(1 + pv.tx) * MP) + (int64_t)(pv.eh + pv.ee) * MP;  // one KV head
    const int64_t per_p = (int64_t)(3 + pv.tx) * T + pv.eh + pv.ee;  // one full M-tile pair
    const int64_t off = it.lo - pv.start[b];
    if (off > 0) {
      // 32-bit divisions when every cost position fits in 32 bits
      const int g = (int)imin64(pv.Hkv - 1, pv.narrow ? (int64_t)((uint32_t)off / (uint32_t)per_g) : off / per_g);
      const int64_t off2 = off - g * per_g;
      const int mp = (int)imin64(MP - 1, pv.narrow ? (int64_t)((uint32_t)off2 / (uint32_t)per_p) : off2 / per_p);
      it.j = g * MP + mp;
      it.gstart = pv.start[b] + g * per_g + (int64_t)mp * per_p;
    }
    if (it.j > 0) {
      const int mpp = (it.j - 1) % MP;
      it.c_prev = imin32(2, MT - 2 * mpp) + 1 + pv.tx;
    } else {
      int bp = b - 1;
      while (bp >= 0 && pv.T[bp] == 0) --bp;
      if (bp >= 0) {
        const int MTp = pv.MT[bp], MPp = (MTp + 1) / 2;
        it.c_prev = imin32(2, MTp - 2 * (MPp - 1)) + 1 + pv.tx;
      }
    }
  }
}

TV_PLAN_FN bool iter_next(ItemIter& it, const PlanView& pv, int cta, Item& o) {
  for (;;) {
    if (it.b >= pv.B || it.gstart >= it.hi) return false;
    const int T = pv.T[it.b];
    const int MT = pv.MT[it.b], MP = (MT + 1) / 2;
    if (T == 0 || it.j >= pv.Hkv * MP) {
      ++it.b;
      it.j = 0;
      continue;
    }
    const int g = it.j / MP, mp = it.j - g * MP;
    const int nt = imin32(2, MT - 2 * mp);
    const int c = nt + 1 + pv.tx;
    const int64_t gs = it.gstart;
    const int64_t t0 = gs + pv.eh;  // the group's first tile
    const int64_t i_lo = imin64(T, ceil_div_c(it.lo - t0, c));
    const int64_t i_hi = imin64(T, ceil_div_c(it.hi - t0, c));
    const int c_prev = it.c_prev;
    it.gstart += (int64_t)T * c + pv.eh + pv.ee;
    it.c_prev = c;
    ++it.j;
    if (i_lo >= i_hi) continue;
    o.b = it.b;
    o.g = g;
    o.mp = mp;
    o.nt = nt;
    o.tile_begin = (int)i_lo;
    o.tile_end = (int)i_hi;
    o.k0 = pv.owner(t0);
    o.n_splits = pv.owner(t0 + (int64_t)(T - 1) * c) - o.k0 + 1;
    // split 0's slot: 2*k0 when the group is CTA k0's first item (the previous
    // group's last tile, ee + c_prev units before gs, is another CTA's), else
    // 2*k0 + 1; every later split is its CTA's first item
    const bool first_of_k0 = (c_prev == 0) || pv.owner(gs - pv.ee - c_prev) < o.k0;
    o.slot0 = 2 * o.k0 + (first_of_k0 ? 0 : 1);
    o.my_slot = 2 * cta + (it.produced == 0 ? 0 : 1);
    ++it.produced;
    return true;
  }
}

// Partial slot of split sp of a group (split 0's slot depends on whether the
// group is its CTA's first item; every later split is its CTA's first item).
TV_PLAN_INL int split_slot(const Item& it, int sp) { return sp == 0 ? it.slot0 : 2 * (it.k0 + sp); }

}  // namespace attn
}  // namespace tv

#endif  // TV_ATTN_PLAN_CUH_
