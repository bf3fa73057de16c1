// tv_tree_verify_attn: tree-masked, split-KV paged attention of a draft tree
// over each request's KV cache, on sm_103a tensor cores, in one launch.
//
// "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2: the whole
// candidate tree (<= 64 nodes) is scored by one forward pass whose attention
// uses the mask M[i][j] = 1 iff j is an ancestor of i or i itself.  Every node
// also sees the request's full prefix.  For query head h, node i:
//   out = softmax(scale * q K_vis^T) V_vis,  lse = ln sum exp(scale * q K_vis^T)
// over the visible keys K_vis = prefix (0..L-1) + {L + j : j in A(i)}.
//
// GB300 mapping
//  * Query rows of one KV head are (node, head-in-group) pairs: row m = i*G + r.
//    128 rows form an M tile; a work group is (request, KV head, M-tile pair),
//    so one K/V tile feeds up to 256 query rows.
//  * K/V pages (16 tokens x D) stream through TMA into 128-byte-swizzled
//    shared memory, 8 pages per 128-key tile, two-stage rings for K and V.
//  * S = Q K^T (SS MMA, K-major) and O += P V (TS MMA: P in TMEM, V MN-major)
//    run on tcgen05 with fp32 accumulators in TMEM: S_t at columns t*128,
//    O_t at 256 + t*D; P (bf16 pairs) overwrites the S columns it came from.
//  * Warp roles: warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM owner,
//    warp 3 planner and page-table checker, warps 4-7 / 8-11 softmax and
//    epilogue of M tile 0 / 1 (one row per thread, tcgen05.ld 32x32b).
//    Online softmax in base 2 with a lazy rescale of O (only when the row max
//    grows by more than 2^8).
//  * The ancestor mask enters as one 32-bit visibility word per 32 keys:
//    prefix keys are all visible, tree key L+j is visible iff bit j of the
//    row's 64-bit ancestor word is set, keys past L+N are not.
//  * Work division: every CTA computes the same plan from the request lengths
//    and takes an equal share of the total (KV tile x M tile) cost, contiguous
//    in (request, KV head, M-tile pair, KV tile) order.  A group cut between
//    CTAs is a split: each split writes a normalised partial and its
//    log-sum-exp, takes a ticket, and the last split to arrive merges them.
//    Nothing waits on another CTA.
//  * All roles walk the same item sequence; reuse of Q, K/V stages and the O
//    accumulators between items is ordered by mbarriers, so the next item's
//    loads overlap the current item's epilogue.
//  * Request errors found on the device (bad page id, timeout) are collected
//    in the workspace; the last CTA to exit folds them into `status` and
//    zero-fills those requests, so no CTA's plan reads a status bit written
//    during the same launch.  Every wait is bounded (about one second).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include "attn_common.cuh"

namespace tv {
namespace attn {

// Plan cost units charged at each end of a work group, on top of nt + 1 units
// per KV tile: the item's epilogue and the restart of its pipeline cost about as
// much as a few tiles, so a CTA that crosses more group boundaries takes fewer
// tiles (serving batch 140 -> 112 us, 7B shape 22.3 -> 20.7 us against no charge).
constexpr int kItemEnd = 6;
// Low-bit cache: a KV tile costs its decode, which does not grow with the active
// M tiles, so the plan charges each tile kTileDecode units more (in units of the
// bf16 kernel's per-tile cost nt + 1; serving batch, 4-bit: 146.7 / 135.1 / 134.9 /
// 149.5 us at 0 / 1 / 2 / 4 units).
constexpr int kTileDecode = 2;
constexpr int kItemEndQ4 = 6;

// dynamic shared-memory layout (1024-byte aligned base)
template <int D, int kLB>
struct Smem {
  static constexpr bool kQ4 = kLB != 0;                   // a low-bit (4- or 3-bit) cache
  static constexpr int kDBlocks = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr int kQTile = kBM * D * 2;
  static constexpr int kKVTile = kBN * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kNT * kQTile;
  static constexpr int kV = kK + kStages * kKVTile;
  // low-bit cache: for K and for V two code slots of half a tile each, a slot
  // holding the codes [64 keys][D/2 or 3D/8] followed by the params [64 keys][D/16] fp16
  static constexpr int kCodeRow = kLB == 3 ? 3 * D / 8 : D / 2;
  static constexpr int kParamRow = D / 8;
  static constexpr int kSlotParams = kHalfKeys * kCodeRow;
  static constexpr int kSlot = kHalfKeys * (kCodeRow + kParamRow);
  static constexpr int kKC = kV + kStages * kKVTile;
  static constexpr int kVC = kKC + (kQ4 ? 2 * kSlot : 0);
  static constexpr int kMB = kQ4 ? kMaxBatchQ4 : kMaxBatch;
  static constexpr int kRqStart = kVC + (kQ4 ? 2 * kSlot : 0);   // int64 [kMB + 1]
  static constexpr int kRqT = kRqStart + 8 * (kMB + 1) + 8;      // int32 [kMB]
  static constexpr int kRqMT = kRqT + 4 * kMB;                   // int32 [kMB]
  static constexpr int kBytes = kRqMT + 4 * kMB;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc + 2048 <= 227 * 1024, "shared memory over the per-CTA limit");
};


template <int D, int kLB>
__device__ __forceinline__ void merge_tile(const AttnParams& p, const Item& it, int mtile, int n_rows, int r) {
  // (splits per round trip, 16-byte loads per split): about 128 registers of loads
  // and accumulators either way; half of that where the launch leaves 128 registers
  // a thread (4-bit cache)
  const int mrow0 = (it.mp * kNT + mtile) * kBM, prow0 = mtile * kBM;
  auto slot_of = [&](int sp) { return split_slot(it, sp); };
  if constexpr (kLB != 0) {
    if (it.n_splits <= 2) merge_items<D, 2, (D >= 128 ? 4 : 2), kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else if (it.n_splits <= 4) merge_items<D, 4, 2, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else if (it.n_splits <= 6) merge_items<D, 6, 2, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else merge_items<D, 8, 1, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
  } else {
    if (it.n_splits <= 2) merge_items<D, 2, (D >= 128 ? 8 : 4), kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else if (it.n_splits <= 4) merge_items<D, 4, 4, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else if (it.n_splits <= 6) merge_items<D, 6, 4, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
    else merge_items<D, 8, 2, kBM>(p, it, mrow0, prow0, n_rows, r, slot_of);
  }
}

// One key row of a low-bit code slot, held in registers: the decoding thread
// copies its row out and frees the slot for the next tile's codes before it
// decodes, so that load overlaps this tile's decode.  4-bit: each 32-dim group's
// 32 codes (one 16-byte word) and its (scale, zero) fp16 pair, scale in the low
// half.  3-bit: each group's two words of low bits and one word of third bits.
template <int D, int kLB>
struct CodeRow {
  static constexpr int kGroups = D / kQ4Group;
  uint4 c[kGroups];      // 4-bit: the group's codes; 3-bit: x, y low bits, z third bits
  uint32_t pw[kGroups];
};

// Copies row `codes` / `params` of a code slot.  4-bit rows are 64 bytes apart,
// so a quarter-warp's 16-byte loads of one group would hit the same four banks
// four times: rows 2i and 2i + 1 start at group i mod 4 (entry k holds group
// (k + rot) mod 4).  3-bit rows are 48 bytes apart and need no rotation.
template <int D, int kLB>
__device__ __forceinline__ void load_code_row(CodeRow<D, kLB>& x, const uint8_t* codes, const uint8_t* params,
                                              int rot) {
  constexpr int kG = CodeRow<D, kLB>::kGroups;
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const int gi = (k + rot) & (kG - 1);
    if constexpr (kLB == 3) {
      const uint2 l = reinterpret_cast<const uint2*>(codes)[gi];
      x.c[k] = make_uint4(l.x, l.y, reinterpret_cast<const uint32_t*>(codes + D / 4)[gi], 0u);
    } else {
      x.c[k] = reinterpret_cast<const uint4*>(codes)[gi];
    }
    x.pw[k] = reinterpret_cast<const uint32_t*>(params)[gi];
  }
}

// Decodes a code row into key row r of a bf16 K or V stage, laid out as the TMA
// copies of a bf16 cache are (64-dim blocks of 128-byte rows, 16-byte chunks
// swizzled by the row's low three bits).  Dim d of the row takes the value
// bf16(fp32(code * scale + zero)) with the (scale, zero) pair of its 32-dim group.
// 4-bit codes: byte j of a group holds dim 2j in its low nibble and 2j + 1 in its
// high nibble.  3-bit codes: the row's low two bits four per byte (byte j: dims
// 4j .. 4j+3, dim 4j+i in bits 2i and 2i+1), then its third bits eight per byte
// (byte D/4 + j: dims 8j .. 8j+7, dim 8j+i in bit i); four codes at a time are
// spread into the bytes of a word, the low-bit pairs by shifts of 6, 12 and 18
// (each lands at the bottom of its own byte), the third bits by a multiply with
// 1 + 2^7 + 2^14 + 2^21 (bit k lands at bit 8k).  A code (4-bit: a whole byte of
// two codes, split in fp32 below) becomes a float exactly by placing it in the
// low mantissa bits of 2^23 and subtracting 2^23; the fused multiply-add then
// rounds the exact code * scale + zero once to fp32, and the conversion rounds
// that once to bf16.
// The groups are a loop, not unrolled (each turn selects its group's registers
// by compare, so every register index is fixed): the decoding warps share each SM
// sub-partition's instruction cache with the softmax, and an unrolled row
// (about 500 instructions) ran 15-20% slower.
template <int D, int kLB>
__device__ __forceinline__ void decode_code_row(const CodeRow<D, kLB>& x, uint8_t* stage, int r, int rot) {
  constexpr int kG = CodeRow<D, kLB>::kGroups;
  const uint64_t neg_magic = f2_pack(-8388608.f, -8388608.f);
#pragma unroll 1
  for (int k = 0; k < kG; ++k) {
    const int gi = (k + rot) & (kG - 1);
    uint4 c = x.c[0];
    uint32_t pw = x.pw[0];
#pragma unroll
    for (int u = 1; u < kG; ++u)
      if (k == u) {
        c = x.c[u];
        pw = x.pw[u];
      }
    const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&pw));
    const uint64_t s2 = f2_pack(sz.x, sz.x), z2 = f2_pack(sz.y, sz.y);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // dims 8q .. 8q + 7 of the group: one 16-byte chunk
      uint32_t cw[2];  // 3-bit: codes of dims 8q .. 8q+3 and 8q+4 .. 8q+7, one per byte
      if constexpr (kLB == 3) {
        const uint32_t l16 = (q < 2 ? c.x : c.y) >> (16 * (q & 1));
        const uint32_t h8 = c.z >> (8 * q);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t b = (l16 >> (8 * u)) & 0xFFu;
          const uint32_t lb = (b | (b << 6) | (b << 12) | (b << 18)) & 0x03030303u;
          const uint32_t hb = (((h8 >> (4 * u)) & 0xFu) * 0x00204081u) & 0x01010101u;
          cw[u] = lb | (hb << 2);
        }
      }
      uint32_t o[4];
      if constexpr (kLB == 3) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float ce = __uint_as_float(__byte_perm(cw[j >> 1], 0x4B000000u, 0x7440u + 2 * (j & 1)));
          const float co = __uint_as_float(__byte_perm(cw[j >> 1], 0x4B000000u, 0x7440u + 2 * (j & 1) + 1));
          float ve, vo;
          f2_unpack(f2_fma(f2_add(f2_pack(ce, co), neg_magic), s2, z2), ve, vo);
          o[j] = pack_bf16x2(ve, vo);
        }
      } else {
        // A whole byte b = low + 16 high becomes 2^23 + b, then the nibbles are split
        // in fp32, exactly: (b - 7.5) / 16 + 1.5 * 2^23 lies within 15/32 of
        // 1.5 * 2^23 + high, where the spacing of fp32 is 1, so it rounds to that
        // (no ties); low = b - 16 high.  This takes half the byte permutes and none
        // of the nibble masks of a permute per code.
        const uint32_t w = q == 0 ? c.x : q == 1 ? c.y : q == 2 ? c.z : c.w;
        const uint64_t m75 = f2_pack(-7.5f, -7.5f), r16 = f2_pack(0.0625f, 0.0625f);
        const uint64_t big = f2_pack(12582912.f, 12582912.f), nbig = f2_pack(-12582912.f, -12582912.f);
        const uint64_t n16 = f2_pack(-16.f, -16.f);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {  // bytes 2 pr and 2 pr + 1 of the word: dims 4 pr .. 4 pr + 3
          const float fa = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + 2 * pr));
          const float fb = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + 2 * pr + 1));
          const uint64_t b = f2_add(f2_pack(fa, fb), neg_magic);  // the two bytes
          const uint64_t hn = f2_add(f2_fma(f2_add(b, m75), r16, big), nbig);  // their high nibbles
          const uint64_t ln = f2_fma(hn, n16, b);                               // their low nibbles
          float l0, l1, h0, h1;
          f2_unpack(f2_fma(ln, s2, z2), l0, l1);
          f2_unpack(f2_fma(hn, s2, z2), h0, h1);
          o[2 * pr] = pack_bf16x2(l0, h0);
          o[2 * pr + 1] = pack_bf16x2(l1, h1);
        }
      }
      const int d0 = gi * kQ4Group + q * 8;
      const int db = d0 / 64, ch = (d0 % 64) / 8;
      *reinterpret_cast<uint4*>(stage + db * (kBN * 128) + r * 128 + ((ch ^ (r & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <int D, int kLB>
__global__ void __launch_bounds__(kLB != 0 ? kThreadsQ4 : kThreads, 1)
    verify_attn_kernel(const __grid_constant__ AttnParams p) {
  using S = Smem<D, kLB>;
  constexpr bool kQ4 = kLB != 0;  // a low-bit cache, decoded by warps 12-19
  constexpr int kNThreads = kQ4 ? kThreadsQ4 : kThreads;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_qe, bar_kf[kStages], bar_ke[kStages], bar_vf[kStages], bar_ve[kStages];
  __shared__ uint64_t bar_s[kNT], bar_p[kNT], bar_o[kNT], bar_of[kNT], bar_wg[kNT], bar_ml;
  // 4-bit cache: code slots full / free (K and V), one pair per half tile
  __shared__ uint64_t bar_kcf[2], bar_kce[2], bar_vcf[2], bar_vce[2];
  // low-bit cache: pages of the tile whose codes a slot holds (-1: no more tiles),
  // written by the producer before it fills the slot
  __shared__ int slot_npg[2][2];
  __shared__ float ml_sh[2][kBM];  // dual mode: warpgroup 1's running max and sum per row
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ int64_t plan_W;
  __shared__ int plan_C;
  __shared__ int ticket_sh[kNT];
  __shared__ int last_cta_sh;
  __shared__ int last_b_sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cta = blockIdx.x;
  int64_t* rq_start = reinterpret_cast<int64_t*>(smem + S::kRqStart);
  int32_t* rq_T = reinterpret_cast<int32_t*>(smem + S::kRqT);
  int32_t* rq_MT = reinterpret_cast<int32_t*>(smem + S::kRqMT);

  if (tid == 0) {
    abort_sh = 0;
    last_b_sh = -1;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qe, 1);
    for (int s = 0; s < kStages; ++s) {
      // a bf16 stage is filled by TMA (one arrival plus bytes) or by 128 decoding threads
      mbar_init(&bar_kf[s], kQ4 ? kBN : 1);
      mbar_init(&bar_ke[s], 1);
      mbar_init(&bar_vf[s], kQ4 ? kBN : 1);
      mbar_init(&bar_ve[s], 1);
    }
    if (kQ4) {
      for (int h = 0; h < 2; ++h) {
        mbar_init(&bar_kcf[h], 1);
        mbar_init(&bar_kce[h], kHalfKeys);
        mbar_init(&bar_vcf[h], 1);
        mbar_init(&bar_vce[h], kHalfKeys);
      }
    }
    for (int t = 0; t < kNT; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], kBM);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_of[t], kBM);
      mbar_init(&bar_wg[t], kBM);
    }
    mbar_init(&bar_ml, kBM);
    fence_barrier_init();
  }
  if (warp == 0) {
    tma_prefetch_desc(&p.tmQ);
    if (!kQ4) {
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
    }
  }
  if (warp == 2) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  // Nothing that a call starting its successor early writes is read before the wait
  // on the previous kernel: the plan reads the request lengths, the producers Q, the
  // cache and the page table (so the first tiles load over the previous kernel's
  // tail), the MMA issuer and the decoders only on-chip memory.  The softmax and
  // the page-table check, which read the masks and write outputs and workspace,
  // wait at their first item (after_previous), and the exit path waits before the
  // workspace.  A request flagged in `status` (which the previous kernel may write)
  // is computed like any other and zero-filled at exit.
  if (warp == 3) {
    // ---- plan: per-request tiles and costs, exclusive scan of the costs
    int64_t carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int64_t cost = 0;
      if (b < p.B) {
        const int L = p.prefix_len[b], N = p.n_nodes[b];
        const bool skip = request_shape_bits(L, N, p.n_max, p.max_pages) != 0;
        int T = 0, MT = 0;
        if (!skip) {
          T = (L + N + kBN - 1) / kBN;
          MT = (N * p.G + kBM - 1) / kBM;
          constexpr int kTx = kQ4 ? kTileDecode : 0, kEnd = kQ4 ? kItemEndQ4 : kItemEnd;
          cost = (int64_t)p.Hkv * ((int64_t)T * (MT + (1 + kTx) * ((MT + 1) / 2)) + 2ll * kEnd * ((MT + 1) / 2));
        }
        rq_T[b] = T;
        rq_MT[b] = MT;
      }
      int64_t incl = cost;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < p.B) rq_start[b] = carry + incl - cost;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      rq_start[p.B] = carry;
      plan_W = carry;
      // at least one tile's cost (3 + tx units at most) per CTA, so that every CTA
      // between a group's first and last split holds a tile of it
      plan_C = (int)imax64(1, imin64(gridDim.x, carry / (3 + (kQ4 ? kTileDecode : 0))));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  PlanView pv;
  pv.start = rq_start;
  pv.T = rq_T;
  pv.MT = rq_MT;
  pv.B = p.B;
  pv.Hkv = p.Hkv;
  pv.eh = kQ4 ? kItemEndQ4 : kItemEnd;
  pv.ee = kQ4 ? kItemEndQ4 : kItemEnd;
  pv.tx = kQ4 ? kTileDecode : 0;
  pv.W = plan_W;
  pv.C = plan_C;
  pv.narrow = (int64_t)(plan_C + 1) * plan_W < (int64_t(1) << 32);
  const bool has_work = pv.W > 0 && cta < pv.C;

  uint8_t* sQ = smem + S::kQ;
  uint8_t* sK = smem + S::kK;
  uint8_t* sV = smem + S::kV;
  const int G = p.G;

  if (has_work && (warp == 0 || warp == 2)) {
    // ------------------------------------------------------------ TMA producers
    // warp 0 loads Q and the K stages, warp 2 the V stages: a V stage waits for the
    // PVs of the stage it replaces, which must not hold back later K stages
    setmaxnreg_dec<kQ4 ? kRegsControlQ4 : kRegsControl>();
    const bool is_k = warp == 0;
    if (elect_one_sync()) {
      ItemIter it;
      iter_init(it, pv, cta);
      Item item;
      uint32_t kv_it = 0, n_item = 0;
      const int qrows_per_tile = p.q_box_nodes * G;
      bool ok = true;
      while (ok && iter_next(it, pv, cta, item)) {
        if (is_k) {
          // Q of the previous item is free once its last QK^T has completed
          if (n_item > 0) ok = mbar_wait(&bar_qe, (n_item - 1) & 1u, &abort_sh);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_q, (uint32_t)(item.nt * S::kDBlocks * qrows_per_tile * 128));
          const int node0 = item.mp * kNT * (kBM / G);
          for (int t = 0; t < item.nt; ++t)
            for (int db = 0; db < S::kDBlocks; ++db)
              tma_load_4d(sQ + t * S::kQTile + db * (kBM * 128), &p.tmQ, &bar_q, db * 64, item.g * G,
                          node0 + t * (kBM / G), item.b);
        }
        const int L = p.prefix_len[item.b], N = p.n_nodes[item.b];
        const int32_t* pt = p.page_table + (int64_t)item.b * p.max_pages;
        for (int tile = item.tile_begin; tile < item.tile_end && ok; ++tile, ++kv_it) {
          const int key0 = tile * kBN;
          const int npg = min(kPagesPerTile, (L + N - key0 + kPageSize - 1) / kPageSize);
          int pages[kPagesPerTile];
#pragma unroll
          for (int pg = 0; pg < kPagesPerTile; ++pg) pages[pg] = pg < npg ? pt[key0 / kPageSize + pg] : 0;
          if constexpr (kQ4) {
            // codes and params of each half tile into its code slot (bulk copies of the
            // contiguous per-page blocks); an out-of-range page id reads page 0 instead
            // (the request is reported and zero-filled at exit)
            const uint8_t* codes = is_k ? p.k_codes : p.v_codes;
            const uint8_t* prm = is_k ? p.k_params : p.v_params;
            constexpr uint32_t kPgCodes = kPageSize * S::kCodeRow, kPgParams = kPageSize * S::kParamRow;
            for (int h = 0; h < 2 && ok; ++h) {
              uint64_t* cfree = is_k ? &bar_kce[h] : &bar_vce[h];
              uint64_t* cfull = is_k ? &bar_kcf[h] : &bar_vcf[h];
              uint8_t* slot = smem + (is_k ? S::kKC : S::kVC) + h * S::kSlot;
              ok = mbar_wait(cfree, (kv_it & 1u) ^ 1u, &abort_sh);
              if (!ok) break;
              const int pg0 = h * (kPagesPerTile / 2);
              const int n_pg = max(0, min(kPagesPerTile / 2, npg - pg0));
              slot_npg[is_k ? 0 : 1][h] = npg;
              mbar_arrive_expect_tx(cfull, (uint32_t)n_pg * (kPgCodes + kPgParams));
              for (int i = 0; i < n_pg; ++i) {
                int id = pages[pg0 + i];
                if (id < 0 || (int64_t)id >= p.num_pages) id = 0;
                const int64_t blk = (int64_t)id * p.Hkv + item.g;
                bulk_g2s(slot + i * kPgCodes, codes + blk * kPgCodes, kPgCodes, cfull);
                bulk_g2s(slot + S::kSlotParams + i * kPgParams, prm + blk * kPgParams, kPgParams, cfull);
              }
            }
          } else {
            // an out-of-range page id reads the TMA fill value (zeros); the request is
            // reported and zero-filled at exit
            const int s = kv_it % kStages;
            const uint32_t ph = (kv_it / kStages) & 1u;
            const uint32_t bytes = (uint32_t)(npg * kPageSize * D * 2);
            uint64_t* empty = is_k ? &bar_ke[s] : &bar_ve[s];
            uint64_t* full = is_k ? &bar_kf[s] : &bar_vf[s];
            uint8_t* dst = (is_k ? sK : sV) + s * S::kKVTile;
            const CUtensorMap* map = is_k ? &p.tmK : &p.tmV;
            ok = mbar_wait(empty, ph ^ 1u, &abort_sh);
            if (!ok) break;
            mbar_arrive_expect_tx(full, bytes);
            for (int pg = 0; pg < npg; ++pg)
              for (int db = 0; db < S::kDBlocks; ++db)
                tma_load_4d(dst + db * (kBN * 128) + pg * (kPageSize * 128), map, full, db * 64, 0, item.g,
                            pages[pg]);
          }
        }
        ++n_item;
      }
      if constexpr (kQ4) {
        // no more tiles: the decoders of each half find -1 in their slot's page count
        for (int h = 0; h < 2 && ok; ++h) {
          ok = mbar_wait(is_k ? &bar_kce[h] : &bar_vce[h], (kv_it & 1u) ^ 1u, &abort_sh);
          if (!ok) break;
          slot_npg[is_k ? 0 : 1][h] = -1;
          mbar_arrive(is_k ? &bar_kcf[h] : &bar_vcf[h]);
        }
      }
    }
    __syncwarp();
  } else if (has_work && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    setmaxnreg_dec<kQ4 ? kRegsControlQ4 : kRegsControl>();
    if (elect_one_sync()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, false, true);
      // Descriptors of the operand bases; an operand offset is added to the start
      // address field (bytes / 16), so each MMA costs one add and the issue keeps
      // pace with the tensor pipe.
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      // S_t = Q_qt K^T for the K stage in slot s (128 keys)
      auto issue_qk = [&](int t, int qt, int s) {
        const uint32_t d = tmem + t * 128;
        const uint64_t a = dq0 + (uint64_t)((qt * S::kQTile) >> 4);
        const uint64_t b = dk0 + (uint64_t)((s * S::kKVTile) >> 4);
#pragma unroll
        for (int db = 0; db < S::kDBlocks; ++db)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, a + (uint64_t)((db * (kBM * 128) + kk * 32) >> 4),
                   b + (uint64_t)((db * (kBN * 128) + kk * 32) >> 4), idesc_qk, (db | kk) != 0);
      };
      // O_t (+)= P_t V   (P_t is packed bf16 over the S_t columns)
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint32_t d = tmem + 256 + t * D;
        const uint64_t b = dv0 + (uint64_t)((s * S::kKVTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(d, tmem + t * 128 + kk * 8, b + (uint64_t)((kk * 2048) >> 4), idesc_pv, (acc || kk > 0) ? 1u : 0u);
      };
      ItemIter it;
      iter_init(it, pv, cta);
      Item item;
      uint32_t kv_it = 0, n_item = 0;
      uint32_t ph_p[kNT] = {0, 0};
      uint32_t uses[kNT] = {0, 0};  // items that used accumulator t so far
      bool ok = true;
      while (ok && iter_next(it, pv, cta, item)) {
        const int n_tiles = item.tile_end - item.tile_begin;
        // one active M tile over several KV stages: the two softmax warpgroups take
        // alternate stages, each with its own S and O (combined in the epilogue)
        const bool dual = item.nt == 1 && n_tiles >= 2;
        const int n_wg = dual ? 2 : item.nt;
        const int nu0 = dual ? (n_tiles + 1) / 2 : n_tiles;             // stages of warpgroup 0
        const int nu1 = dual ? n_tiles / 2 : (item.nt == 2 ? n_tiles : 0);  // stages of warpgroup 1
        const int per_stage = dual ? 1 : item.nt;  // warpgroups reading one stage
        int kf_next = 0, vf_next = 0;              // next stage whose K / V arrival is awaited
        int qk_cnt = 0, pv_cnt = 0;                // warpgroups done with the oldest unreleased stage
        int qk_rel = 0, pv_rel = 0;                // oldest unreleased K / V stage
        int qk_left = nu0 + nu1;
        auto slot = [&](int j) { return (int)((kv_it + j) % kStages); };
        auto sph = [&](int j) { return ((kv_it + j) / kStages) & 1u; };
        auto need_k = [&](int j) {
          while (ok && kf_next <= j) {
            ok = mbar_wait(&bar_kf[slot(kf_next)], sph(kf_next), &abort_sh);
            ++kf_next;
          }
          tc_fence_after();
        };
        auto need_v = [&](int j) {
          while (ok && vf_next <= j) {
            ok = mbar_wait(&bar_vf[slot(vf_next)], sph(vf_next), &abort_sh);
            ++vf_next;
          }
          tc_fence_after();
        };
        // stages are read in order (warpgroup 0 first in each round), so the stage
        // to release is always the oldest unreleased one
        auto qk = [&](int t, int k) {
          const int j = dual ? 2 * k + t : k;
          need_k(j);
          if (!ok) return;
          issue_qk(t, dual ? 0 : t, slot(j));
          mma_commit(&bar_s[t]);
          if (++qk_cnt == per_stage) {
            mma_commit(&bar_ke[slot(qk_rel)]);
            ++qk_rel;
            qk_cnt = 0;
          }
          if (--qk_left == 0) mma_commit(&bar_qe);  // the item's last QK^T is issued
        };
        ok = mbar_wait(&bar_q, n_item & 1u, &abort_sh);
        if (ok) qk(0, 0);
        if (ok && nu1 > 0) qk(1, 0);
        for (int k = 0; k < nu0 && ok; ++k) {
          for (int t = 0; t < n_wg && ok; ++t) {
            const int nu = t == 0 ? nu0 : nu1;
            if (k >= nu) continue;
            const int j = dual ? 2 * k + t : k;
            need_v(j);
            // O_t of the previous item must have been read by its epilogue
            if (ok && k == 0 && uses[t] > 0) ok = mbar_wait(&bar_of[t], (uses[t] - 1) & 1u, &abort_sh);
            ok = ok && mbar_wait(&bar_p[t], ph_p[t], &abort_sh);
            ph_p[t] ^= 1u;
            tc_fence_after();
            if (!ok) break;
            issue_pv(t, slot(j), k > 0);
            if (++pv_cnt == per_stage) {
              mma_commit(&bar_ve[slot(pv_rel)]);
              ++pv_rel;
              pv_cnt = 0;
            }
            // S_t of the next stage overwrites P_t after the PV above has read it
            if (k + 1 < nu) qk(t, k + 1);
            else mma_commit(&bar_o[t]);
          }
        }
        for (int t = 0; t < n_wg; ++t) ++uses[t];
        kv_it += n_tiles;
        ++n_item;
      }
    }
    __syncwarp();
  } else if (has_work && warp == 3) {
    // ------------------------------------------------------------ page-table check
    setmaxnreg_dec<kQ4 ? kRegsControlQ4 : kRegsControl>();
    // every needed page of each request this CTA touches
    ItemIter it;
    iter_init(it, pv, cta);
    Item item;
    int prev_b = -1;
    bool waited = false;
    while (iter_next(it, pv, cta, item)) {
      after_previous(waited);
      if (item.b == prev_b) continue;
      prev_b = item.b;
      const int L = p.prefix_len[item.b], N = p.n_nodes[item.b];
      const int need = (L + N + kPageSize - 1) / kPageSize;
      const int32_t* pt = p.page_table + (int64_t)item.b * p.max_pages;
      bool bad = false;
      for (int k = lane; k < need; k += 32) bad |= (pt[k] < 0 || (int64_t)pt[k] >= p.num_pages);
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.ws_bits + item.b, TV_DEV_PAGE_OOB);
    }
  } else if (kQ4 && has_work && warp >= 12) {
    // ------------------------------------------------------------ low-bit decoders
    // warps 12-15 decode K, warps 16-19 V: thread i takes key row i of each tile
    // (rows 0-63 from code slot 0, rows 64-127 from code slot 1)
    setmaxnreg_dec<kRegsDecodeQ4>();
    const bool is_k = warp < 16;
    const int ri = tid - (is_k ? 384 : 512);
    const int h = ri / kHalfKeys;
    const uint8_t* const slot = smem + (is_k ? S::kKC : S::kVC) + h * S::kSlot;
    const uint8_t* const crow = slot + (ri % kHalfKeys) * S::kCodeRow;
    const uint8_t* const prow = slot + S::kSlotParams + (ri % kHalfKeys) * S::kParamRow;
    const int rot = kLB == 3 ? 0 : (ri >> 1) & (D / kQ4Group - 1);  // see load_code_row
    uint64_t* const cfull = is_k ? &bar_kcf[h] : &bar_vcf[h];
    uint64_t* const cfree = is_k ? &bar_kce[h] : &bar_vce[h];
    uint8_t* const stage0 = is_k ? sK : sV;
    // tiles in the producer's order; each slot names its tile's page count
    for (uint32_t kv_it = 0;; ++kv_it) {
      const int s = kv_it % kStages;
      const uint32_t ph = (kv_it / kStages) & 1u;
      if (!warp_wait(cfull, kv_it & 1u, &abort_sh)) break;
      const int npg = slot_npg[is_k ? 0 : 1][h];
      if (npg < 0) break;
      // the row's codes into registers, and the slot back to the producer
      const bool live = ri < npg * kPageSize;
      CodeRow<D, kLB> row;
      if (live) load_code_row<D, kLB>(row, crow, prow, rot);
      // the slot's next bulk copy (async proxy) must not overtake these reads
      fence_proxy_async_smem();
      mbar_arrive(cfree);
      // the bf16 stage is free once the MMAs of the tile it held have completed
      if (!warp_wait(is_k ? &bar_ke[s] : &bar_ve[s], ph ^ 1u, &abort_sh)) break;
      if (live) decode_code_row<D, kLB>(row, stage0 + s * S::kKVTile, ri, rot);
      fence_proxy_async_smem();  // the tensor pipe reads what these threads wrote
      mbar_arrive(is_k ? &bar_kf[s] : &bar_vf[s]);
    }
  } else if (has_work && warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    if constexpr (!kQ4) setmaxnreg_inc<kRegsSoftmax>();
    else setmaxnreg_inc<kRegsSoftmaxQ4>();
    const int t = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;                 // row of the M tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * D;
    const uint32_t tO1 = tmem + lane_base + 256 + D;     // accumulator 1 (read by warpgroup 0 in dual mode)
    const float sl2 = p.scale_log2;
    ItemIter it;
    iter_init(it, pv, cta);
    Item item;
    uint32_t kv_it = 0;
    uint32_t ph_s = 0, ph_o = 0, ph_ml = 0, ph_wg = 0;
    bool ok = true;
    // warpgroup-wide barrier with a bounded wait
    auto wg_sync = [&]() -> bool {
      mbar_arrive(&bar_wg[t]);
      const bool k = warp_wait(&bar_wg[t], ph_wg, &abort_sh);
      ph_wg ^= 1u;
      return k;
    };
    bool waited = false;
    while (ok && iter_next(it, pv, cta, item)) {
      after_previous(waited);
      const int n_tiles = item.tile_end - item.tile_begin;
      const bool dual = item.nt == 1 && n_tiles >= 2;
      if (!dual && t >= item.nt) {
        kv_it += n_tiles;
        continue;
      }
      const int n_units = dual ? (n_tiles - t + 1) / 2 : n_tiles;  // stages of this warpgroup
      if (tid == 128) last_b_sh = item.b;
      const int L = p.prefix_len[item.b];
      const int N = p.n_nodes[item.b];
      const int mtile = dual ? 0 : t;                     // M tile whose rows this warpgroup holds
      const int mrow = (item.mp * kNT + mtile) * kBM + r;
      const int node = mrow / G;
      const int hh = mrow - node * G;
      const bool row_ok = node < N;
      // only bits of the request's own nodes count: a stray bit j >= N in the caller's
      // word would otherwise expose position L + j, which holds no node of this tree
      const uint64_t valid_bits = N >= 64 ? ~0ull : ((1ull << N) - 1ull);
      const uint64_t anc = row_ok ? p.anc_mask[(int64_t)item.b * p.n_max + node] & valid_bits : 0ull;
      float m_run = -INFINITY, l_run = 0.f;
      for (int k = 0; k < n_units; ++k) {
        const int j = dual ? 2 * k + t : k;                       // stage of this unit
        ok = warp_wait(&bar_s[t], ph_s, &abort_sh);
        ph_s ^= 1u;
        tc_fence_after();
        if (!ok) break;
        const int key0 = (item.tile_begin + j) * kBN;             // first key of the stage
        // S values of invisible keys become -inf
        auto mask_keys = [&](uint32_t* x, int n, int k0) {
          if (k0 + n > L) {
#pragma unroll
            for (int c0 = 0; c0 < n; c0 += 32) {
              const uint32_t vis = visible32(k0 + c0, L, anc);
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vis >> c) & 1u)) x[c0 + c] = __float_as_uint(-INFINITY);
            }
          }
        };
        // row max of n values as four independent partial maxima of three-input steps
        auto row_max = [&](const uint32_t* x, int n) {
          float pm[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) pm[u] = fmaxf(__uint_as_float(x[2 * u]), __uint_as_float(x[2 * u + 1]));
#pragma unroll
          for (int c = 8; c < n; c += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              pm[u] = fmax3(pm[u], __uint_as_float(x[c + 2 * u]), __uint_as_float(x[c + 2 * u + 1]));
          return fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
        };
        // 128 values of the row (bf16 cache), or 64 at a time for the maximum (4-bit
        // cache: the row is read again in chunks of 32 for its probabilities)
        constexpr int kW = kQ4 ? kBN / 2 : kBN;
        uint32_t v[kW];
        float mx;
        if constexpr (kQ4) {
          tmem_ld64(tS, v);
          mask_keys(v, 64, key0);
          const float mx0 = row_max(v, 64);
          tmem_ld64(tS + 64, v);
          mask_keys(v, 64, key0 + 64);
          mx = fmaxf(mx0, row_max(v, 64));
        } else {
          tmem_ld128(tS, v);
          mask_keys(v, kBN, key0);
          mx = row_max(v, kBN);
        }
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool grow = m_new > m_run + kRescaleLog2;
        const float alpha = grow ? ex2_approx(m_run - m_new) : 1.f;  // 0 when m_run = -inf
        if (grow) {
          l_run *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        // a stage that runs past the request's data: clear its V rows past the data
        // (before the first PV that reads this stage)
        if ((dual || t == 0) && key0 + kBN > L + N) {
          const uint32_t kk = kv_it + j;
          const int s = kk % kStages;
          ok = warp_wait(&bar_vf[s], (kk / kStages) & 1u, &abort_sh);
          if (!ok) break;
          const int vr = L + N - key0;
          uint8_t* vbase = sV + s * S::kKVTile;
          const int nch = (kBN - vr) * 8 * S::kDBlocks;
          for (int q = r; q < nch; q += kBM) {
            const int db = q % S::kDBlocks;
            const int rest = q / S::kDBlocks;
            *reinterpret_cast<uint4*>(vbase + db * (kBN * 128) + (vr + rest / 8) * 128 + (rest % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // probabilities 2^(s*scale*log2e - m), packed in place as bf16 pairs; the
        // scaling and the row sum run two lanes per instruction
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m_use, -m_use);
        uint64_t ps2[2] = {0ull, 0ull};
        auto exps = [&](uint32_t* x, int n) {
#pragma unroll
          for (int c = 0; c < n; c += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c]), __uint_as_float(x[c + 1])), sl2x2, negm2), x0, x1);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            ps2[(c >> 1) & 1] = f2_add(ps2[(c >> 1) & 1], f2_pack(e0, e1));
            x[c >> 1] = pack_bf16x2(e0, e1);
          }
        };
        if constexpr (kQ4) {
          // chunk c of 32 keys: its P (16 packed columns) goes to columns 16c.., all
          // of which were read before (the layout the bf16 path writes in one step)
#pragma unroll 1
          for (int c0 = 0; c0 < kBN; c0 += 32) {
            uint32_t x[32];
            tmem_ld32(tS + c0, x);
            mask_keys(x, 32, key0 + c0);
            exps(x, 32);
            tmem_st16(tS + c0 / 2, x);
          }
        } else {
          exps(v, kBN);
          tmem_st64(tS, v);
        }
        float ps[4];
        f2_unpack(ps2[0], ps[0], ps[1]);
        f2_unpack(ps2[1], ps[2], ps[3]);
        const float rs = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        if (__any_sync(0xffffffffu, grow && k > 0)) {
          // rescale O (the PV of this accumulator's previous stage completed before the
          // S of this stage became ready; the next PV waits for this thread's arrival)
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c0, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(tO + c0, o);
          }
        }
        l_run += rs;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar_p[t]);
      }
      kv_it += n_tiles;
      if (!ok) break;
      // ---- epilogue
      ok = warp_wait(&bar_o[t], ph_o, &abort_sh);
      ph_o ^= 1u;
      tc_fence_after();
      if (!ok) break;
      float m_c = m_run, l_c = l_run, a0 = 1.f, a1 = 0.f;
      if (dual) {
        if (t == 1) {
          // hand the row state to warpgroup 0, which combines both accumulators
          ml_sh[0][r] = m_run;
          ml_sh[1][r] = l_run;
          tc_fence_before();
          mbar_arrive(&bar_ml);
          continue;
        }
        ok = warp_wait(&bar_ml, ph_ml, &abort_sh);
        ph_ml ^= 1u;
        tc_fence_after();
        if (!ok) break;
        const float m1 = ml_sh[0][r], l1 = ml_sh[1][r];
        m_c = fmaxf(m_run, m1);
        const float mu = (m_c == -INFINITY) ? 0.f : m_c;
        a0 = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - mu);
        a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - mu);
        l_c = l_run * a0 + l1 * a1;
      }
      const float inv_l = l_c > 0.f ? 1.f / l_c : 0.f;
      const float lse_v = l_c > 0.f ? (m_c + __log2f(l_c)) * 0.69314718055994531f : -INFINITY;
      const int h = item.g * G + hh;
      const int64_t orow_idx = ((int64_t)item.b * p.n_max + node) * p.Hq + h;
      const bool direct = item.n_splits == 1;
      const int prow = mtile * kBM + r;
      // the normalised row (both accumulators in dual mode), in chunks of 32 columns
      auto row_chunk = [&](int c0, float* y) {
        uint32_t o[32];
        tmem_ld32(tO + c0, o);
        if (dual) {
          uint32_t o1[32];
          tmem_ld32(tO1 + c0, o1);
#pragma unroll
          for (int c = 0; c < 32; ++c) y[c] = (__uint_as_float(o[c]) * a0 + __uint_as_float(o1[c]) * a1) * inv_l;
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(o[c]) * inv_l;
        }
      };
      // a partial row is stored as fp16 values of O / c: c = 1, or c = max |O| for a row
      // with a value past the fp16 range (found on the way; that row is stored again)
      uint4* pslot = p.part_o + (int64_t)item.my_slot * (D / 8) * kRowsPerSlot + prow;
      auto half_store = [&](const float* y, int c0, float sc) {
        uint4* dst = pslot + (c0 / 8) * kRowsPerSlot;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 h = __floats2half2_rn(y[8 * q + 2 * e] * sc, y[8 * q + 2 * e + 1] * sc);
            hw[e] = *reinterpret_cast<const uint32_t*>(&h);
          }
          dst[q * kRowsPerSlot] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
      };
      float amax = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float y[32];
        row_chunk(c0, y);
        if (direct) {
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow_idx * D + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(y[8 * q], y[8 * q + 1]), pack_bf16x2(y[8 * q + 2], y[8 * q + 3]),
                                  pack_bf16x2(y[8 * q + 4], y[8 * q + 5]), pack_bf16x2(y[8 * q + 6], y[8 * q + 7]));
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) amax = fmaxf(amax, fabsf(y[c]));
          if (row_ok) half_store(y, c0, 1.f);
        }
      }
      constexpr float kHalfMax = 65504.f;
      float row_scale = 1.f;
      if (!direct && __any_sync(0xffffffffu, amax > kHalfMax)) {
        const bool over = amax > kHalfMax;
        if (over) row_scale = amax;
        const float to_half = 1.f / row_scale;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float y[32];
          row_chunk(c0, y);
          if (row_ok && over) half_store(y, c0, to_half);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_of[t]);  // the accumulator(s) may be overwritten by the next item
      if (dual) mbar_arrive(&bar_of[1]);
      if (direct) {
        if (row_ok && p.lse) p.lse[orow_idx] = lse_v;
      } else {
        if (row_ok) {
          p.part_lse[(int64_t)item.my_slot * kRowsPerSlot + prow] = lse_v;
          p.part_scale[(int64_t)item.my_slot * kRowsPerSlot + prow] = row_scale;
        }
        // ticket: the last split of this (group, M tile) to arrive merges every partial.
        // The warpgroup barrier orders every thread's partial stores before the ticket,
        // whose release (GPU scope) covers them; its acquire, passed on by the second
        // barrier, covers the other splits' stores for the merge.
        ok = wg_sync();
        if (!ok) break;
        const int tick_idx = (((item.b * p.Hkv + item.g) * p.mp_max + item.mp) * kNT) + mtile;
        if (r == 0) ticket_sh[t] = atom_add_acq_rel_gpu(p.ws_tickets + tick_idx, 1);
        ok = wg_sync();
        if (!ok) break;
        if (ticket_sh[t] == item.n_splits - 1) {
          const int n_rows = min(kBM, N * G - (item.mp * kNT + mtile) * kBM);  // valid rows of the M tile
          merge_tile<D, kLB>(p, item, mtile, n_rows, r);
          if (r == 0) p.ws_tickets[tick_idx] = 0;  // ready for the next call
        }
      }
    }
  }

  // ---------------------------------------------------------------- exit
  // (a no-op for the threads that waited at their first item)
  griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
  if (tid == 0) {
    if (abort_sh && last_b_sh >= 0) atomicOr(p.ws_bits + last_b_sh, TV_DEV_TIMEOUT);
    // the barrier above orders this CTA's stores before the count, whose release
    // covers them; the last CTA's acquire (passed on by the barrier below) covers all
    last_cta_sh = (atom_add_acq_rel_gpu(p.ws_exit, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (last_cta_sh) finish_requests<D>(p, tid, kNThreads);
}

// ---------------------------------------------------------------- host side
struct WsLayout {
  size_t bits, tickets, exit, part_lse, part_scale, part_o, total;
  int mp_max;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int B, int n_max, int Hq, int Hkv, int D, int grid) {
  WsLayout w;
  const int G = Hq / Hkv;
  const int mt_max = (n_max * G + kBM - 1) / kBM;
  w.mp_max = (mt_max + kNT - 1) / kNT;
  w.exit = 0;
  w.bits = 256;
  w.tickets = align256(w.bits + sizeof(int32_t) * (size_t)std::max(B, 1));
  w.part_lse = align256(w.tickets + sizeof(int32_t) * (size_t)std::max(B, 1) * Hkv * w.mp_max * kNT);
  w.part_scale = align256(w.part_lse + sizeof(float) * (size_t)2 * grid * kRowsPerSlot);
  w.part_o = align256(w.part_scale + sizeof(float) * (size_t)2 * grid * kRowsPerSlot);
  w.total = align256(w.part_o + sizeof(uint16_t) * (size_t)2 * grid * kRowsPerSlot * D);
  return w;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

static bool make_map4(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides[3],
                      const uint32_t box[4]) {
  auto enc = encode_fn();
  if (!enc) return false;
  const uint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kLB>
static int launch(const AttnParams& ap, int grid, cudaStream_t st) {
  using S = Smem<D, kLB>;
  TV_CUDA_CHECK(ensure_smem_attr((const void*)verify_attn_kernel<D, kLB>, S::kAlloc));
  TV_CUDA_CHECK(check_launch_regs((const void*)verify_attn_kernel<D, kLB>, (int)(kLB != 0 ? kRegsLaunchQ4 : kRegsLaunch)));
  TV_CUDA_CHECK(launch_pdl(verify_attn_kernel<D, kLB>, dim3(grid), dim3(kLB != 0 ? kThreadsQ4 : kThreads),
                           (size_t)S::kAlloc, st, ap));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}

// Kernel choice for the bf16 cache: the CTA-pair kernel runs 256 query rows of
// a KV head per pair of SMs, so it pays off when a KV head has at least two such
// blocks (n_max * G >= 512, e.g. 64-node trees with 8 query heads per KV head);
// fewer rows per KV head (MHA, small trees) run one CTA per SM with its own
// 256-row M-tile pairs.  Head dim 64 always runs one CTA per SM.
static int launch_bf16(const AttnParams& ap, int D, int n_max, int grid, cudaStream_t st) {
  if (D == 128 && n_max * ap.G >= 2 * 2 * kBM && n_max * ap.G <= 8 * kBM) return launch_pair(ap, grid, st);
  return D == 128 ? launch<128, 0>(ap, grid, st) : launch<64, 0>(ap, grid, st);
}

// Argument checks and parameter set-up shared by the entry points.
// With low_bits set (4 or 3), k_cache and v_cache are the code arrays and the
// params arrays come in k_params / v_params; no tensor map is made for them.
static int prepare(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                   const int32_t* page_table, int max_pages, const int32_t* prefix_len, const int32_t* n_nodes,
                   const uint64_t* anc_mask, int B, int n_max, int Hq, int Hkv, int D, int page_size, float scale,
                   void* out, float* lse, int32_t* status, AttnParams* ap, int low_bits = 0,
                   const void* k_params = nullptr, const void* v_params = nullptr) {
  const bool q4 = low_bits != 0;
  TV_REQUIRE(q && k_cache && v_cache && page_table && prefix_len && n_nodes && anc_mask && out && status,
             TV_ERR_INVALID_ARG, "tv_tree_verify_attn: NULL pointer");
  TV_REQUIRE(!q4 || (k_params && v_params), TV_ERR_INVALID_ARG, "tv_tree_verify_attn_q%d: NULL params pointer",
             low_bits);
  TV_REQUIRE(!q4 || (aligned16(k_params) && aligned16(v_params)), TV_ERR_INVALID_ARG,
             "tv_tree_verify_attn_q%d: params must be 16-byte aligned", low_bits);
  TV_REQUIRE(!q4 || B <= kMaxBatchQ4, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn_q%d: B = %d not in [0, %d]",
             low_bits, B, kMaxBatchQ4);
  TV_REQUIRE(page_size == kPageSize, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: page_size %d != 16", page_size);
  TV_REQUIRE(D == 64 || D == 128, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: D = %d not in {64, 128}", D);
  TV_REQUIRE(Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0, TV_ERR_UNSUPPORTED,
             "tv_tree_verify_attn: Hq = %d not a multiple of Hkv = %d", Hq, Hkv);
  const int G = Hq / Hkv;
  TV_REQUIRE(G <= kBM && kBM % G == 0, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: group size %d must divide 128", G);
  TV_REQUIRE(n_max >= 1 && n_max <= kMaxNodes, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: n_max = %d not in [1, 64]",
             n_max);
  TV_REQUIRE(B >= 0 && B <= kMaxBatch, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: B = %d not in [0, %d]", B,
             kMaxBatch);
  TV_REQUIRE(num_pages >= 1 && num_pages < (1ll << 31) && max_pages >= 1, TV_ERR_INVALID_ARG,
             "tv_tree_verify_attn: bad page counts");
  TV_REQUIRE(scale > 0.f && std::isfinite(scale), TV_ERR_INVALID_ARG, "tv_tree_verify_attn: scale must be > 0");
  TV_REQUIRE(aligned16(q) && aligned16(k_cache) && aligned16(v_cache) && aligned16(out), TV_ERR_INVALID_ARG,
             "tv_tree_verify_attn: q, caches and out must be 16-byte aligned");
  memset(ap, 0, sizeof(*ap));
  const int q_box_nodes = std::min(kBM / G, n_max);
  if (B > 0) {
    {
      const uint64_t dims[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)n_max, (uint64_t)B};
      const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)n_max * Hq * D * 2};
      const uint32_t box[4] = {64, (uint32_t)G, (uint32_t)q_box_nodes, 1};
      TV_REQUIRE(make_map4(&ap->tmQ, q, dims, str, box), TV_ERR_CUDA, "tv_tree_verify_attn: tensor map for q failed");
    }
    if (!q4) {
      const uint64_t dims[4] = {(uint64_t)D, (uint64_t)kPageSize, (uint64_t)Hkv, (uint64_t)num_pages};
      const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)kPageSize * D * 2, (uint64_t)Hkv * kPageSize * D * 2};
      const uint32_t box[4] = {64, (uint32_t)kPageSize, 1, 1};
      TV_REQUIRE(make_map4(&ap->tmK, k_cache, dims, str, box) && make_map4(&ap->tmV, v_cache, dims, str, box),
                 TV_ERR_CUDA, "tv_tree_verify_attn: tensor map for the KV cache failed");
    }
  }
  if (q4) {
    ap->k_codes = static_cast<const uint8_t*>(k_cache);
    ap->v_codes = static_cast<const uint8_t*>(v_cache);
    ap->k_params = static_cast<const uint8_t*>(k_params);
    ap->v_params = static_cast<const uint8_t*>(v_params);
  }
  ap->q = static_cast<const uint16_t*>(q);
  ap->page_table = page_table;
  ap->prefix_len = prefix_len;
  ap->n_nodes = n_nodes;
  ap->anc_mask = anc_mask;
  ap->out = static_cast<uint16_t*>(out);
  ap->lse = lse;
  ap->status = status;
  ap->num_pages = num_pages;
  ap->B = B;
  ap->max_pages = max_pages;
  ap->n_max = n_max;
  ap->Hq = Hq;
  ap->Hkv = Hkv;
  ap->G = G;
  ap->q_box_nodes = q_box_nodes;
  ap->scale_log2 = (float)((double)scale * 1.4426950408889634);
  return TV_OK;
}

static void bind_workspace(AttnParams* ap, const WsLayout& wl, uint8_t* wsb) {
  ap->ws_exit = reinterpret_cast<int32_t*>(wsb + wl.exit);
  ap->ws_bits = reinterpret_cast<int32_t*>(wsb + wl.bits);
  ap->ws_tickets = reinterpret_cast<int32_t*>(wsb + wl.tickets);
  ap->part_lse = reinterpret_cast<float*>(wsb + wl.part_lse);
  ap->part_scale = reinterpret_cast<float*>(wsb + wl.part_scale);
  ap->part_o = reinterpret_cast<uint4*>(wsb + wl.part_o);
  ap->mp_max = wl.mp_max;
}

}  // namespace attn
}  // namespace tv

extern "C" size_t tv_tree_verify_attn_workspace(int B, int n_max, int Hq, int Hkv, int D, int max_kv_len) {
  (void)max_kv_len;
  if (B < 0 || n_max < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (D != 64 && D != 128)) return 0;
  return tv::attn::ws_layout(B, n_max, Hq, Hkv, D, tv::current_sm_count()).total;
}

extern "C" int tv_tree_verify_attn(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                                   const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                                   const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq,
                                   int Hkv, int D, int page_size, float scale, void* out, float* lse, void* ws,
                                   size_t ws_bytes, int32_t* status, void* stream) {
  using namespace tv::attn;
  tv::clear_error();
  AttnParams ap;
  const int rc = prepare(q, k_cache, v_cache, num_pages, page_table, max_pages, prefix_len, n_nodes, anc_mask, B,
                         n_max, Hq, Hkv, D, page_size, scale, out, lse, status, &ap);
  if (rc != TV_OK) return rc;
  if (B == 0) return TV_OK;
  const int grid = tv::current_sm_count();
  const WsLayout wl = ws_layout(B, n_max, Hq, Hkv, D, grid);
  TV_REQUIRE(ws != nullptr && ws_bytes >= wl.total, TV_ERR_WORKSPACE,
             "tv_tree_verify_attn: workspace %zu bytes < %zu", ws_bytes, wl.total);
  TV_REQUIRE(tv::aligned16(ws), TV_ERR_INVALID_ARG, "tv_tree_verify_attn: workspace must be 16-byte aligned");
  bind_workspace(&ap, wl, static_cast<uint8_t*>(ws));
  cudaStream_t st = tv::as_stream(stream);
  return launch_bf16(ap, D, n_max, grid, st);
}

namespace tv {
namespace attn {
// The low-bit entry points: argument checks, workspace, the decoding kernel.
static int verify_attn_lowbit(int bits, const void* q, const uint8_t* k_codes, const void* k_params,
                              const uint8_t* v_codes, const void* v_params, int64_t num_pages,
                              const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                              const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq, int Hkv,
                              int D, int page_size, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                              int32_t* status, void* stream) {
  clear_error();
  AttnParams ap;
  const int rc = prepare(q, k_codes, v_codes, num_pages, page_table, max_pages, prefix_len, n_nodes, anc_mask, B,
                         n_max, Hq, Hkv, D, page_size, scale, out, lse, status, &ap, bits, k_params, v_params);
  if (rc != TV_OK) return rc;
  if (B == 0) return TV_OK;
  const int grid = current_sm_count();
  const WsLayout wl = ws_layout(B, n_max, Hq, Hkv, D, grid);
  TV_REQUIRE(ws != nullptr && ws_bytes >= wl.total, TV_ERR_WORKSPACE,
             "tv_tree_verify_attn_q%d: workspace %zu bytes < %zu", bits, ws_bytes, wl.total);
  TV_REQUIRE(aligned16(ws), TV_ERR_INVALID_ARG, "tv_tree_verify_attn_q%d: workspace must be 16-byte aligned", bits);
  bind_workspace(&ap, wl, static_cast<uint8_t*>(ws));
  cudaStream_t st = as_stream(stream);
  if (bits == 3) return D == 128 ? launch<128, 3>(ap, grid, st) : launch<64, 3>(ap, grid, st);
  return D == 128 ? launch<128, 4>(ap, grid, st) : launch<64, 4>(ap, grid, st);
}
}  // namespace attn
}  // namespace tv

extern "C" int tv_tree_verify_attn_q4(const void* q, const uint8_t* k_codes, const void* k_params,
                                      const uint8_t* v_codes, const void* v_params, int64_t num_pages,
                                      const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                                      const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq,
                                      int Hkv, int D, int page_size, float scale, void* out, float* lse, void* ws,
                                      size_t ws_bytes, int32_t* status, void* stream) {
  return tv::attn::verify_attn_lowbit(4, q, k_codes, k_params, v_codes, v_params, num_pages, page_table, max_pages,
                                      prefix_len, n_nodes, anc_mask, B, n_max, Hq, Hkv, D, page_size, scale, out,
                                      lse, ws, ws_bytes, status, stream);
}

extern "C" int tv_tree_verify_attn_q3(const void* q, const uint8_t* k_codes, const void* k_params,
                                      const uint8_t* v_codes, const void* v_params, int64_t num_pages,
                                      const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                                      const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq,
                                      int Hkv, int D, int page_size, float scale, void* out, float* lse, void* ws,
                                      size_t ws_bytes, int32_t* status, void* stream) {
  return tv::attn::verify_attn_lowbit(3, q, k_codes, k_params, v_codes, v_params, num_pages, page_table, max_pages,
                                      prefix_len, n_nodes, anc_mask, B, n_max, Hq, Hkv, D, page_size, scale, out,
                                      lse, ws, ws_bytes, status, stream);
}

// ---------------------------------------------------------------- built-in scratch variant
// For callers that cannot allocate device memory themselves, a variant of
// tv_tree_verify_attn runs on a fixed scratch array compiled into this file.
// Every device that loads the library holds the array until the process exits.
namespace tv {
namespace attn {

constexpr size_t kFixedScratchBytes = size_t(48) << 20;  // 48 MiB
static __device__ __align__(256) uint8_t g_fixed_scratch[kFixedScratchBytes];

// Device address of g_fixed_scratch in the current context.  In host code the
// array's name only stands in for the symbol, so its address is looked up with
// the device current and cached per device together with the id of the context
// it was found in.  A device reset (or any other new context on the device)
// loads the library's module again, possibly at another address: a changed
// context id makes the next call look the address up again instead of using the
// old context's pointer.
static int fixed_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  TV_CUDA_CHECK(cudaGetDevice(&dev));
  TV_REQUIRE(dev >= 0 && dev < 64, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn_noalloc: device id %d >= 64", dev);
  unsigned long long ctx_id = 0;
  TV_REQUIRE(current_context_id(&ctx_id) == cudaSuccess, TV_ERR_CUDA,
             "tv_tree_verify_attn_noalloc: the current context could not be queried");
  std::lock_guard<std::mutex> lock(mu);
  if (ctx_id == 0 || addr[dev] == nullptr || ctx_of[dev] != ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fixed_scratch);  // sets up the context if needed
    TV_REQUIRE(e == cudaSuccess && p != nullptr, TV_ERR_CUDA,
               "tv_tree_verify_attn_noalloc: cudaGetSymbolAddress of the built-in scratch failed: %s",
               cudaGetErrorString(e));
    TV_REQUIRE(current_context_id(&ctx_id) == cudaSuccess && ctx_id != 0, TV_ERR_CUDA, "tv_tree_verify_attn_noalloc: no current CUDA context");
    addr[dev] = p;
    ctx_of[dev] = ctx_id;
  }
  *out = addr[dev];
  return TV_OK;
}

}  // namespace attn
}  // namespace tv

extern "C" int tv_tree_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                           int64_t num_pages, const int32_t* page_table, int max_pages,
                                           const int32_t* prefix_len, const int32_t* n_nodes,
                                           const uint64_t* anc_mask, int B, int n_max, int Hq, int Hkv, int D,
                                           int page_size, float scale, void* out, float* lse, int32_t* status,
                                           void* stream) {
  using namespace tv::attn;
  tv::clear_error();
  AttnParams ap;
  const int rc = prepare(q, k_cache, v_cache, num_pages, page_table, max_pages, prefix_len, n_nodes, anc_mask, B,
                         n_max, Hq, Hkv, D, page_size, scale, out, lse, status, &ap);
  if (rc != TV_OK) return rc;
  if (B == 0) return TV_OK;
  const int grid = tv::current_sm_count();
  const WsLayout wl = ws_layout(B, n_max, Hq, Hkv, D, grid);
  TV_REQUIRE(wl.total <= kFixedScratchBytes, TV_ERR_UNSUPPORTED,
             "tv_tree_verify_attn_noalloc: these sizes need %zu bytes of scratch but the built-in scratch holds "
             "%zu; call tv_tree_verify_attn with a workspace instead",
             wl.total, kFixedScratchBytes);
  void* ws = nullptr;
  const int arc = fixed_scratch_address(&ws);
  if (arc != TV_OK) return arc;
  cudaStream_t st = tv::as_stream(stream);
  // the array keeps the previous call's contents (possibly of other sizes):
  // clear the counters and error bits the kernel expects to start at zero
  TV_CUDA_CHECK(cudaMemsetAsync(ws, 0, wl.part_lse, st));
  bind_workspace(&ap, wl, static_cast<uint8_t*>(ws));
  return launch_bf16(ap, D, n_max, grid, st);
}
