// tv_tree_verify_attn on CTA pairs: the same tree-masked split-KV attention as
// verify_attn.cu ("SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2:
// one forward pass over the candidate tree with the ancestor mask M, every node
// also seeing the request's prefix), laid out for head dim 128 on two SMs at a
// time.
//
// GB300 mapping
//  * A cluster of two CTAs runs one group of 256 query rows (rows m = i*G + r
//    of one KV head: CTA rank k holds rows 128k .. 128k + 127) with
//    tcgen05.mma.cta_group::2: each M = 256 MMA is issued once by CTA 0 and
//    runs on both SMs' tensor cores, each reading its own rows of A and writing
//    its own rows of D, and half of the B operand from its own shared memory.
//  * S = Q K^T reads Q and K from shared memory; O += P V reads P from TMEM
//    (written over the S columns it came from) and V from shared memory.  K
//    and V stream in halves: CTA k loads keys 64k .. 64k + 63 of each 128-key
//    tile (QK's N split) and dims 64k .. 64k + 63 of V (PV's N split), so each
//    SM holds 32 KB per K/V stage and the rings are four stages deep.  Both
//    CTAs' copies of a stage (and of Q) count on CTA 0's barrier, which CTA 0's
//    producer arms with the bytes of both halves.  The last, partial tile of a
//    request is the exception: each CTA's V half counts on its own barrier, its
//    softmax threads clear the V rows past the data, and their arrival on CTA
//    0's P barrier tells the MMA thread that the half is ready.
//  * The group's KV tiles alternate between two accumulator chains, each with
//    its own S and O in TMEM (S0 S1 O0 O1: all 512 columns) and its own softmax
//    warpgroup (one row per thread).  The QK^T of stage k + 2 is issued right
//    after the PV of stage k, so one chain's softmax runs while the other
//    chain's MMAs keep the tensor pipe busy; the epilogue combines the two
//    chains by their row maxima and sums.  Online softmax in base 2 against a
//    reference max that a chain's first stage sets and later stages keep while
//    their probabilities stay below 2^32 (checked on the row sum, no max pass);
//    a stage that would pass it raises the reference and rescales O (rare).
//    Both warpgroups take the epilogue of every item, each half of O's
//    columns, after swapping their row states; a split's merge runs on both.
//  * Work division: block c of every KV head runs on the clusters of lane c;
//    within a lane the plan of verify_attn.cu splits the (request, KV head,
//    KV tile) sequence evenly over its clusters, so the lanes read each K/V
//    tile at about the same time (one read from DRAM, the others from L2).
//    Split groups merge per CTA half.
//  * Every wait is bounded (about one second); on a timeout the kernel unwinds
//    and reports TV_DEV_TIMEOUT for the request, as the one-CTA kernel does.
#include <algorithm>
#include <mutex>
#include "attn_common.cuh"

namespace tv {
namespace attn {

constexpr int kPD = 128;            // head dim of this kernel
constexpr int kPStages = 4;         // K and V ring depth (half tiles)
constexpr int kPThreads = 384;      // 12 warps
constexpr int kPHalfKeys = 64;      // keys of this CTA's K half tile
constexpr uint32_t kWgArrivals = 8; // one arrival per warp of a softmax warpgroup, from both CTAs
constexpr uint32_t kEpArrivals = 16;  // one arrival per softmax warp of both warpgroups, from both CTAs
constexpr int kMaxLanes = 4;        // 256-row blocks per KV head (n_max * G <= 1024)
// Plan cost units charged at the start and at the end of a (request, KV head)
// group, on top of 3 units per KV tile: the restart of an item's two chains,
// its epilogue and a split's merge take about as long as a few stages, so a
// cluster that crosses more group boundaries gets fewer tiles.
// (Charging the ends differently, 2-8 units at the start and 12-16 at the end,
// measured the same on the 70B and long-context batches.)
constexpr int kPairItemStart = 8, kPairItemEnd = 8;

struct PairSmem {
  static constexpr int kQTile = kBM * kPD * 2;          // [2 dim blocks][128 rows][128 B]
  static constexpr int kKStage = kPHalfKeys * kPD * 2;  // [2 dim blocks][64 keys][128 B]
  static constexpr int kVStage = kBN * 64 * 2;          // [128 keys][128 B]: this CTA's 64 dims
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQTile;
  static constexpr int kV = kK + kPStages * kKStage;
  static constexpr int kRqStart = kV + kPStages * kVStage;  // int64 [kMaxBatch + 1]
  static constexpr int kRqT = kRqStart + 8 * (kMaxBatch + 1) + 8;
  static constexpr int kRqMT = kRqT + 4 * kMaxBatch;
  static constexpr int kBytes = kRqMT + 4 * kMaxBatch;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc + 4096 <= 227 * 1024, "shared memory over the per-CTA limit");
};

// Partial slot of this CTA for slot s of its lane's plan (plan slots count the
// lane's clusters from lane_base; each CTA of the pair keeps its own rows in its
// own slot).
__device__ __forceinline__ int pair_ws_slot(int lane_base, int s, uint32_t rank) {
  return ((lane_base + (s >> 1)) * 2 + (int)rank) * 2 + (s & 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    verify_attn_pair_kernel(const __grid_constant__ AttnParams p) {
  using S = PairSmem;
  constexpr int D = kPD;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_qe;                        // CTA 0: both Q halves landed; Q free again
  __shared__ uint64_t bar_kf[kPStages], bar_vf[kPStages];  // CTA 0: both halves of the stage landed
  __shared__ uint64_t bar_ke[kPStages], bar_ve[kPStages];  // stage free again (MMA commit, both CTAs)
  __shared__ uint64_t bar_s[kNT], bar_p[kNT], bar_o[kNT], bar_of[kNT], bar_ep;
  __shared__ float ml_sh[2][2][kBM];  // [warpgroup][running max, sum][row]: the chains' row states
  __shared__ float amax_sh[2][kBM];   // [warpgroup][row]: largest |O| of the warpgroup's columns
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ int64_t plan_W;
  __shared__ int plan_C, plan_lane, plan_base;
  __shared__ int ticket_sh[kNT];
  __shared__ int last_cta_sh;
  __shared__ int last_b_sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1;  // the plan's worker: one per cluster
  const int n_cl = gridDim.x >> 1;
  int64_t* rq_start = reinterpret_cast<int64_t*>(smem + S::kRqStart);
  int32_t* rq_T = reinterpret_cast<int32_t*>(smem + S::kRqT);
  int32_t* rq_MT = reinterpret_cast<int32_t*>(smem + S::kRqMT);

  if (tid == 0) {
    abort_sh = 0;
    last_b_sh = -1;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qe, 1);
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&bar_kf[s], 1);
      mbar_init(&bar_vf[s], 1);
      mbar_init(&bar_ke[s], 1);
      mbar_init(&bar_ve[s], 1);
    }
    for (int t = 0; t < kNT; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], kWgArrivals);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_of[t], kEpArrivals);
    }
    mbar_init(&bar_ep, 2 * kBM);
    fence_barrier_init();
  }
  if (warp == 0) {
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
  }
  if (warp == 2) {
    tmem_alloc2(&tmem_sh, 512);
    tmem_relinquish2();
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
    // ---- plan.  Block c (query rows 256c .. 256c + 255) of every (request, KV head)
    // belongs to lane c; each lane gets a share of the clusters proportional to its
    // cost, and within a lane the clusters split the (request, KV head, KV tile)
    // sequence evenly (the one-CTA plan with one 256-row "M-tile pair" per KV head).
    // The lanes walk the same sequence at the same pace, so the blocks of one KV
    // head read each K/V tile at about the same time and all but one read come
    // from L2.
    // pass 1: lane costs (every tile costs 3 units, as a pair of M tiles does)
    int64_t wl[kMaxLanes];
#pragma unroll
    for (int l = 0; l < kMaxLanes; ++l) wl[l] = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int64_t cost = 0;
      int chains = 0;
      if (b < p.B) {
        const int L = p.prefix_len[b], N = p.n_nodes[b];
        const bool skip = request_shape_bits(L, N, p.n_max, p.max_pages) != 0;
        if (!skip) {
          cost = (int64_t)p.Hkv * (((L + N + kBN - 1) / kBN) * 3 + kPairItemStart + kPairItemEnd);
          chains = (N * p.G + 2 * kBM - 1) / (2 * kBM);
        }
      }
#pragma unroll
      for (int l = 0; l < kMaxLanes; ++l) {
        int64_t c = (l < p.mp_max && chains > l) ? cost : 0;
#pragma unroll
        for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        wl[l] += c;
      }
    }
    // clusters of each lane: one for every lane with work, the rest by cost
    int64_t w_all = 0;
    int nz = 0;
#pragma unroll
    for (int l = 0; l < kMaxLanes; ++l) {
      w_all += wl[l];
      nz += wl[l] > 0;
    }
    const int spare = max(0, n_cl - nz);
    int my_lane = -1, lane_base = 0, lane_cl = 0, first = 0;
#pragma unroll
    for (int l = 0; l < kMaxLanes; ++l) {
      const int cnt = wl[l] > 0 ? 1 + (int)(spare * wl[l] / imax64(1, w_all)) : 0;
      if (my_lane < 0 && cl >= first && cl < first + cnt) {
        my_lane = l;
        lane_base = first;
        lane_cl = cnt;
      }
      first += cnt;
    }
    // pass 2: this lane's plan (requests whose rows reach block my_lane)
    int64_t carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int64_t cost = 0;
      if (b < p.B) {
        const int L = p.prefix_len[b], N = p.n_nodes[b];
        const bool skip = my_lane < 0 || request_shape_bits(L, N, p.n_max, p.max_pages) != 0 ||
                          (N * p.G + 2 * kBM - 1) / (2 * kBM) <= my_lane;
        const int T = skip ? 0 : (L + N + kBN - 1) / kBN;
        cost = T > 0 ? (int64_t)p.Hkv * (T * 3 + kPairItemStart + kPairItemEnd) : 0;
        rq_T[b] = T;
        rq_MT[b] = 2;
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
      plan_C = (int)imax64(1, imin64(lane_cl, carry / 3));
      plan_lane = my_lane;
      plan_base = lane_base;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  PlanView pv;
  pv.start = rq_start;
  pv.T = rq_T;
  pv.MT = rq_MT;
  pv.B = p.B;
  pv.Hkv = p.Hkv;
  pv.eh = kPairItemStart;
  pv.ee = kPairItemEnd;
  pv.tx = 0;
  pv.W = plan_W;
  pv.C = plan_C;
  pv.narrow = (int64_t)(plan_C + 1) * plan_W < (int64_t(1) << 32);
  const int lane_id = plan_lane;          // this cluster's 256-row block index
  const int wk = cl - plan_base;          // this cluster's worker index within its lane
  const bool has_work = lane_id >= 0 && pv.W > 0 && wk < pv.C;

  uint8_t* sQ = smem + S::kQ;
  uint8_t* sK = smem + S::kK;
  uint8_t* sV = smem + S::kV;
  const int G = p.G;

  if (has_work && (warp == 0 || warp == 2)) {
    // ------------------------------------------------------------ TMA producers
    // warp 0 loads this CTA's Q rows and K halves, warp 2 its V halves; every copy
    // counts on CTA 0's barrier, which CTA 0's producer arms with both halves' bytes
    setmaxnreg_dec<kRegsControl>();
    const bool is_k = warp == 0;
    if (elect_one_sync()) {
      ItemIter it;
      iter_init(it, pv, wk);
      Item item;
      uint32_t kv_it = 0, n_item = 0;
      bool ok = true;
      auto leader = [&](uint64_t* bar) { return mapa_shared(smem_u32(bar), 0); };
      while (ok && iter_next(it, pv, wk, item)) {
        if (is_k) {
          // Q of the previous item is free once its last QK^T has completed
          if (n_item > 0) ok = mbar_wait(&bar_qe, (n_item - 1) & 1u, &abort_sh);
          if (!ok) break;
          const int node0 = (lane_id * 2 * kBM + (int)rank * kBM) / G;
          if (rank == 0) mbar_arrive_expect_tx(&bar_q, (uint32_t)(2 * 2 * p.q_box_nodes * G * 128));
          for (int db = 0; db < 2; ++db)
            tma_load_4d_pair(sQ + db * (kBM * 128), &p.tmQ, leader(&bar_q), db * 64, item.g * G, node0, item.b);
        }
        const int L = p.prefix_len[item.b], N = p.n_nodes[item.b];
        const int32_t* pt = p.page_table + (int64_t)item.b * p.max_pages;
        for (int tile = item.tile_begin; tile < item.tile_end && ok; ++tile, ++kv_it) {
          const int key0 = tile * kBN;
          const int n_data = L + N - key0;                  // keys of the tile that hold data
          const int npg = min(kPagesPerTile, (n_data + kPageSize - 1) / kPageSize);
          const int s = kv_it % kPStages;
          const uint32_t ph = (kv_it / kPStages) & 1u;
          ok = mbar_wait(is_k ? &bar_ke[s] : &bar_ve[s], ph ^ 1u, &abort_sh);
          if (!ok) break;
          // an out-of-range page id reads the TMA fill value (zeros); the request is
          // reported and zero-filled at exit
          if (is_k) {
            // keys past the data are masked by the softmax, so only pages with data load
            auto n_half = [&](int r) { return max(0, min(kPagesPerTile / 2, npg - r * (kPagesPerTile / 2))); };
            const int pg0 = (int)rank * (kPagesPerTile / 2);
            uint8_t* dst = sK + s * S::kKStage;
            if (rank == 0)
              mbar_arrive_expect_tx(&bar_kf[s], (uint32_t)((n_half(0) + n_half(1)) * 2 * kPageSize * 128));
            for (int i = 0; i < n_half((int)rank); ++i) {
              const int page = pt[key0 / kPageSize + pg0 + i];
              for (int db = 0; db < 2; ++db)
                tma_load_4d_pair(dst + db * (kPHalfKeys * 128) + i * (kPageSize * 128), &p.tmK, leader(&bar_kf[s]),
                                 db * 64, 0, item.g, page);
            }
          } else {
            uint8_t* dst = sV + s * S::kVStage;
            if (n_data >= kBN) {
              // a full tile: both halves count on CTA 0's barrier
              if (rank == 0) mbar_arrive_expect_tx(&bar_vf[s], (uint32_t)(2 * kBN * 128));
              for (int pg = 0; pg < kPagesPerTile; ++pg)
                tma_load_4d_pair(dst + pg * (kPageSize * 128), &p.tmV, leader(&bar_vf[s]), (int)rank * 64, 0,
                                 item.g, pt[key0 / kPageSize + pg]);
            } else {
              // the partial last tile: this CTA's half counts on its own barrier (its
              // softmax threads clear the rows past the data before their P arrival)
              mbar_arrive_expect_tx(&bar_vf[s], (uint32_t)(npg * kPageSize * 128));
              for (int pg = 0; pg < npg; ++pg)
                tma_load_4d(dst + pg * (kPageSize * 128), &p.tmV, &bar_vf[s], (int)rank * 64, 0, item.g,
                            pt[key0 / kPageSize + pg]);
            }
          }
        }
        ++n_item;
      }
    }
    __syncwarp();
  } else if (has_work && (warp == 1 || warp == 3) && rank == 1) {
    // CTA 1's MMA and page-check warps have no role (they take part in the register split)
    setmaxnreg_dec<kRegsControl>();
  } else if (has_work && rank == 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    setmaxnreg_dec<kRegsControl>();
    if (elect_one_sync()) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(2 * kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(2 * kBM, D, false, true);
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      ItemIter it;
      iter_init(it, pv, wk);
      Item item;
      uint32_t kv_it = 0, n_item = 0;
      uint32_t ph_p = 0;             // bit t: phase of bar_p[t]
      uint32_t uses[kNT] = {0, 0};   // items that used accumulator t so far
      bool ok = true;
      while (ok && iter_next(it, pv, wk, item)) {
        const int T = item.tile_end - item.tile_begin;
        int kf_next = 0, vf_next = 0;
        auto slot = [&](int j) { return (int)((kv_it + j) % kPStages); };
        auto sph = [&](int j) { return ((kv_it + j) / kPStages) & 1u; };
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
        // S[j & 1] = Q K_j^T over the pair
        auto qk = [&](int j) {
          need_k(j);
          if (!ok) return;
          const uint32_t d = tmem + (uint32_t)(j & 1) * 128;
          const uint64_t b = dk0 + (uint64_t)((slot(j) * S::kKStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma2_ss(d, dq0 + (uint64_t)(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4),
                    b + (uint64_t)(((kk >> 2) * (kPHalfKeys * 128) + (kk & 3) * 32) >> 4), idesc_qk,
                    kk > 0 ? 1u : 0u);
          mma_commit2_mc(&bar_ke[slot(j)], 3);
          mma_commit2_mc(&bar_s[j & 1], 3);
          if (j == T - 1) mma_commit2_mc(&bar_qe, 3);  // the item's last read of Q
        };
        // the item's Q rows are in both CTAs' shared memory
        ok = mbar_wait(&bar_q, n_item & 1u, &abort_sh);
        tc_fence_after();
        if (ok) qk(0);
        if (ok && T > 1) qk(1);
        for (int k = 0; k < T && ok; ++k) {
          const int t = k & 1;
          need_v(k);
          // O_t of the previous item that used it must have been read by its epilogue
          if (ok && k < 2 && uses[t] > 0) ok = mbar_wait(&bar_of[t], (uses[t] - 1) & 1u, &abort_sh);
          ok = ok && mbar_wait(&bar_p[t], (ph_p >> t) & 1u, &abort_sh);
          ph_p ^= 1u << t;
          tc_fence_after();
          if (!ok) break;
          const uint64_t b = dv0 + (uint64_t)((slot(k) * S::kVStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma2_ts(tmem + 256 + (uint32_t)t * D, tmem + (uint32_t)t * 128 + kk * 8, b + (uint64_t)((kk * 2048) >> 4),
                    idesc_pv, (k >= 2 || kk > 0) ? 1u : 0u);
          mma_commit2_mc(&bar_ve[slot(k)], 3);
          // S of stage k + 2 overwrites P of stage k after the PVs above have read it
          if (k + 2 < T) qk(k + 2);
          else mma_commit2_mc(&bar_o[t], 3);  // chain t's last PV of the item
        }
        ++uses[0];
        if (T > 1) ++uses[1];
        kv_it += T;
        ++n_item;
      }
    }
    __syncwarp();
  } else if (has_work && rank == 0 && warp == 3) {
    // ------------------------------------------------------------ page-table check
    setmaxnreg_dec<kRegsControl>();
    ItemIter it;
    iter_init(it, pv, wk);
    Item item;
    int prev_b = -1;
    bool waited = false;
    while (iter_next(it, pv, wk, item)) {
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
  } else if (has_work && warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    // warpgroup t runs chain t: the item's stages k with k % 2 == t (all of them, on
    // chain 0, for a single-stage item); one row per thread
    setmaxnreg_inc<kRegsSoftmax>();
    const int t = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;                 // row of this CTA's 128 = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * D;
    const float sl2 = p.scale_log2;
    ItemIter it;
    iter_init(it, pv, wk);
    Item item;
    uint32_t kv_it = 0;
    uint32_t ph_s = 0, ph_ep = 0;
    uint32_t ph_o[kNT] = {0u, 0u};  // phases of bar_o, waited on by both warpgroups
    uint32_t rag_ph = 0;  // bit s: phase of CTA 1's bar_vf[s] (partial tiles only)
    bool ok = true;
    // one arrival per warp on CTA 0's barrier (after every lane's TMEM writes)
    auto arrive_leader = [&](uint64_t* bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(bar);
        else mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
      }
    };
    // both softmax warpgroups of this CTA (the epilogue is split between them)
    auto ep_sync = [&]() -> bool {
      mbar_arrive(&bar_ep);
      const bool k = warp_wait(&bar_ep, ph_ep, &abort_sh);
      ph_ep ^= 1u;
      return k;
    };
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
    bool waited = false;
    while (ok && iter_next(it, pv, wk, item)) {
      after_previous(waited);
      const int T = item.tile_end - item.tile_begin;
      const bool dual = T >= 2;
      // the item's partial last tile (if any) completes a phase of CTA 1's barrier of
      // its stage slot; both warpgroups keep that phase, whichever processes the tile
      const uint32_t rag_prev = rag_ph;
      if ((int64_t)item.tile_end * kBN > (int64_t)p.prefix_len[item.b] + p.n_nodes[item.b])
        rag_ph ^= 1u << ((kv_it + T - 1) % kPStages);
      // stages of this chain (none for warpgroup 1 on a single-stage item: it only
      // takes its half of the epilogue)
      const int n_units = dual ? (T - t + 1) / 2 : (t == 0 ? T : 0);
      if (tid == 128) last_b_sh = item.b;
      const int L = p.prefix_len[item.b];
      const int N = p.n_nodes[item.b];
      // only bits of the request's own nodes count: a stray bit j >= N in the caller's
      // word would otherwise expose position L + j, which holds no node of this tree
      const uint64_t valid_bits = N >= 64 ? ~0ull : ((1ull << N) - 1ull);
      const int mrow0 = lane_id * 2 * kBM + (int)rank * kBM;  // first row of this CTA's half of the group
      const int mrow = mrow0 + r;
      const int node = mrow / G;
      const int hh = mrow - node * G;
      const bool row_ok = node < N;
      const uint64_t anc = row_ok ? p.anc_mask[(int64_t)item.b * p.n_max + node] & valid_bits : 0ull;
      float m_run = -INFINITY, l_run = 0.f;
      for (int u = 0; u < n_units; ++u) {
        const int k = dual ? 2 * u + t : u;                 // stage of this unit
        ok = warp_wait(&bar_s[t], ph_s, &abort_sh);
        ph_s ^= 1u;
        tc_fence_after();
        if (!ok) break;
        const int key0 = (item.tile_begin + k) * kBN;     // first key of the stage
        // S values of invisible keys become -inf
        auto load_scores = [&](uint32_t* x) {
          tmem_ld128(tS, x);
          if (key0 + kBN > L) {
#pragma unroll
            for (int c0 = 0; c0 < kBN; c0 += 32) {
              const uint32_t vis = visible32(key0 + c0, L, anc);
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vis >> c) & 1u)) x[c0 + c] = __float_as_uint(-INFINITY);
            }
          }
        };
        // probabilities 2^(s*scale*log2e - m) for the reference m, packed in place as
        // bf16 pairs; the scaling and the row sum run two lanes per instruction
        auto exps = [&](uint32_t* x, float m_ref) {
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m_use, -m_use);
          uint64_t ps2[2] = {0ull, 0ull};
#pragma unroll
          for (int c = 0; c < kBN; c += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c]), __uint_as_float(x[c + 1])), sl2x2, negm2), x0, x1);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            ps2[(c >> 1) & 1] = f2_add(ps2[(c >> 1) & 1], f2_pack(e0, e1));
            x[c >> 1] = pack_bf16x2(e0, e1);
          }
          float ps[4];
          f2_unpack(ps2[0], ps[0], ps[1]);
          f2_unpack(ps2[1], ps[2], ps[3]);
          return (ps[0] + ps[1]) + (ps[2] + ps[3]);
        };
        uint32_t v[kBN];
        load_scores(v);
        // The reference max m_run is set by the chain's first stage with a visible key
        // and kept while this stage's probabilities stay below 2^32 (their row sum says
        // so, with no separate max pass); a stage that would reach 2^32 raises it to its
        // own max and rescales the row's sum and O (rare).  Probabilities of any size up
        // to 2^32 keep bf16/fp32 relative precision, and no sum can overflow.
        if (__any_sync(0xffffffffu, m_run == -INFINITY)) {
          const float mx = row_max(v, kBN);
          if (m_run == -INFINITY) m_run = mx * sl2;  // still -inf if every key is invisible
        }
        // the partial last tile: clear this CTA's V rows past the data once its half
        // has landed (before the P arrival that lets the MMA thread read the stage);
        // CTA 1's barrier of a stage completes only for such tiles
        if (key0 + kBN > L + N) {
          const uint32_t kk = kv_it + k;
          const int s = kk % kPStages;
          const uint32_t ph = rank == 0 ? (kk / kPStages) & 1u : (rag_prev >> s) & 1u;
          ok = warp_wait(&bar_vf[s], ph, &abort_sh);
          if (!ok) break;
          const int vr = L + N - key0;
          uint8_t* vbase = sV + s * S::kVStage;
          const int nch = (kBN - vr) * 8;
          for (int q = r; q < nch; q += kBM)
            *reinterpret_cast<uint4*>(vbase + (vr + q / 8) * 128 + (q % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
        float rs = exps(v, m_run);
        const bool over = !(rs < 4294967296.f);  // 2^32, or not finite
        if (__any_sync(0xffffffffu, over)) {
          // re-read the scores (P is not stored yet), move the reference to this stage's
          // max, rescale this chain's sum and O (the PV of its previous stage completed
          // before this stage's S was ready) and recompute
          load_scores(v);
          const float mx = row_max(v, kBN);
          const float m_new = over ? fmaxf(m_run, mx * sl2) : m_run;
          const float alpha = over ? ex2_approx(m_run - m_new) : 1.f;
          l_run *= alpha;
          m_run = m_new;
          if (u > 0) rescale_o<D>(tO, alpha);
          rs = exps(v, m_run);
        }
        tmem_st64(tS, v);
        tmem_st_wait();
        l_run += rs;
        arrive_leader(&bar_p[t]);
      }
      kv_it += T;
      if (!ok) break;
      // ---- epilogue: warpgroup t takes columns 64t .. 64t + 63 of the combined O
      // rows (both chains in dual mode, chain 0 otherwise)
      ok = warp_wait(&bar_o[0], ph_o[0], &abort_sh);
      ph_o[0] ^= 1u;
      if (ok && dual) {
        ok = warp_wait(&bar_o[1], ph_o[1], &abort_sh);
        ph_o[1] ^= 1u;
      }
      tc_fence_after();
      if (!ok) break;
      // the two warpgroups swap their row states
      ml_sh[t][0][r] = m_run;
      ml_sh[t][1][r] = l_run;
      ok = ep_sync();
      if (!ok) break;
      const float m0 = ml_sh[0][0][r], l0 = ml_sh[0][1][r];
      float m_c = m0, l_c = l0, a0 = 1.f, a1 = 0.f;
      if (dual) {
        const float m1 = ml_sh[1][0][r], l1 = ml_sh[1][1][r];
        m_c = fmaxf(m0, m1);
        const float mu = (m_c == -INFINITY) ? 0.f : m_c;
        a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - mu);
        a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - mu);
        l_c = l0 * a0 + l1 * a1;
      }
      const float inv_l = l_c > 0.f ? 1.f / l_c : 0.f;
      const float lse_v = l_c > 0.f ? (m_c + __log2f(l_c)) * 0.69314718055994531f : -INFINITY;
      const int h = item.g * G + hh;
      const int64_t orow_idx = ((int64_t)item.b * p.n_max + node) * p.Hq + h;
      const bool direct = item.n_splits == 1;
      const int my_slot = pair_ws_slot(plan_base, item.my_slot, rank);
      const int col0 = t * (D / 2);
      const uint32_t tO0 = tmem + lane_base + 256, tO1 = tO0 + D;
      // the normalised row, in chunks of 32 columns
      auto row_chunk = [&](int c0, float* y) {
        uint32_t o[32];
        tmem_ld32(tO0 + c0, o);
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
      uint4* pslot = p.part_o + (int64_t)my_slot * (D / 8) * kRowsPerSlot + r;
      auto half_store = [&](const float* y, int c0, float sc) {
        uint4* dst = pslot + (c0 / 8) * kRowsPerSlot;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 hv = __floats2half2_rn(y[8 * q + 2 * e] * sc, y[8 * q + 2 * e + 1] * sc);
            hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          dst[q * kRowsPerSlot] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
      };
      float amax = 0.f;
#pragma unroll 1
      for (int c0 = col0; c0 < col0 + D / 2; c0 += 32) {
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
      if (!direct) {
        // one scale per row for both halves
        amax_sh[t][r] = amax;
        ok = ep_sync();
        if (!ok) break;
        const float row_amax = fmaxf(amax_sh[0][r], amax_sh[1][r]);
        if (__any_sync(0xffffffffu, row_amax > kHalfMax)) {
          const bool over = row_amax > kHalfMax;
          if (over) row_scale = row_amax;
          const float to_half = 1.f / row_scale;
#pragma unroll 1
          for (int c0 = col0; c0 < col0 + D / 2; c0 += 32) {
            float y[32];
            row_chunk(c0, y);
            if (row_ok && over) half_store(y, c0, to_half);
          }
        }
      }
      arrive_leader(&bar_of[0]);  // the accumulator(s) may be overwritten by the next item
      if (dual) arrive_leader(&bar_of[1]);
      if (direct) {
        if (row_ok && t == 0 && p.lse) p.lse[orow_idx] = lse_v;
      } else {
        if (row_ok && t == 0) {
          p.part_lse[(int64_t)my_slot * kRowsPerSlot + r] = lse_v;
          p.part_scale[(int64_t)my_slot * kRowsPerSlot + r] = row_scale;
        }
        // ticket of this CTA's rows: the last split to arrive merges every partial.  The
        // barrier of both warpgroups orders every thread's partial stores before the
        // ticket, whose release (GPU scope) covers them; its acquire, passed on by the
        // second barrier, covers the other splits' stores for the merge.
        ok = ep_sync();
        if (!ok) break;
        const int tick_idx = (((item.b * p.Hkv + item.g) * p.mp_max + lane_id) * kNT) + (int)rank;
        if (t == 0 && r == 0) ticket_sh[0] = atom_add_acq_rel_gpu(p.ws_tickets + tick_idx, 1);
        ok = ep_sync();
        if (!ok) break;
        if (ticket_sh[0] == item.n_splits - 1) {
          const int n_rows = min(kBM, N * G - mrow0);
          if (n_rows > 0) {
            const int r2 = t * kBM + r;  // both warpgroups
            auto slot_of = [&](int sp) { return pair_ws_slot(plan_base, split_slot(item, sp), rank); };
            if (item.n_splits <= 2) merge_items<D, 2, 8, 2 * kBM>(p, item, mrow0, 0, n_rows, r2, slot_of);
            else if (item.n_splits <= 4) merge_items<D, 4, 4, 2 * kBM>(p, item, mrow0, 0, n_rows, r2, slot_of);
            else if (item.n_splits <= 6) merge_items<D, 6, 4, 2 * kBM>(p, item, mrow0, 0, n_rows, r2, slot_of);
            else merge_items<D, 8, 2, 2 * kBM>(p, item, mrow0, 0, n_rows, r2, slot_of);
          }
          if (t == 0 && r == 0) p.ws_tickets[tick_idx] = 0;  // ready for the next call
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
  cluster_sync_all();  // nothing of this CTA is read or signalled by its peer any more
  tc_fence_after();
  if (warp == 2) tmem_dealloc2(tmem, 512);
  if (tid == 0) {
    if (abort_sh && last_b_sh >= 0) atomicOr(p.ws_bits + last_b_sh, TV_DEV_TIMEOUT);
    // the barrier above orders this CTA's stores before the count, whose release
    // covers them; the last CTA's acquire (passed on by the barrier below) covers all
    last_cta_sh = (atom_add_acq_rel_gpu(p.ws_exit, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (last_cta_sh) finish_requests<D>(p, tid, kPThreads);
}

// Clusters of two CTAs that can be resident at once (cached per context).
static int pair_clusters_resident() {
  static std::mutex mu;
  static unsigned long long ctx_of = 0;
  static int known = 0;
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (known > 0 && ctx != 0 && ctx == ctx_of) return known;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * current_sm_count());
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PairSmem::kAlloc;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_attn_pair_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  known = n;
  ctx_of = ctx;
  return n;
}

int launch_pair(const AttnParams& ap, int max_ctas, cudaStream_t st) {
  TV_CUDA_CHECK(ensure_smem_attr((const void*)verify_attn_pair_kernel, PairSmem::kAlloc));
  TV_CUDA_CHECK(check_launch_regs((const void*)verify_attn_pair_kernel, (int)kRegsLaunch));
  const int resident = pair_clusters_resident();
  TV_REQUIRE(resident > 0, TV_ERR_CUDA, "tv_tree_verify_attn: no CTA pair of the attention kernel fits an SM pair");
  const int grid = 2 * std::max(1, std::min(resident, max_ctas / 2));
  TV_CUDA_CHECK(launch_pdl(verify_attn_pair_kernel, dim3(grid), dim3(kPThreads), (size_t)PairSmem::kAlloc, st, ap));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}

}  // namespace attn
}  // namespace tv
