// tv_tree_verify_attn: tree-masked, split-KV paged attention of a draft tree
// over each request's KV cache, on sm_103a tensor cores.
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
//    128 rows form an M tile; a CTA owns up to two M tiles (256 rows) of one
//    (request, KV head), so K/V tiles are read once for 256 rows.
//  * K/V pages (16 tokens x D) stream through TMA into 128-byte-swizzled
//    shared memory, 8 pages per 128-key tile, two-stage ring per operand.
//  * S = Q K^T (SS MMA, K-major) and O += P V (TS MMA: P in TMEM, V MN-major)
//    run on tcgen05 with fp32 accumulators in TMEM: S_t at columns t*128,
//    O_t at 256 + t*D; P (bf16 pairs) overwrites the S columns it came from.
//  * Warp roles: warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM owner,
//    warps 4-7 / 8-11 softmax + epilogue of M tile 0 / 1 (one row per thread,
//    tcgen05.ld 32x32b).  Online softmax in base 2 with a lazy rescale of O
//    (only when the row max grows by more than 2^8).
//  * The ancestor mask is applied from the row's 64-bit word, only on the
//    tile(s) holding keys >= L; prefix tiles run unmasked.
//  * Split-KV: a device-side plan cuts every (request, KV head, M-tile pair)
//    into key ranges of similar cost; persistent CTAs take work items from an
//    atomic counter; split rows are merged by log-sum-exp weights afterwards.
//  * Every wait is bounded (about one second); on expiry the request gets
//    TV_DEV_TIMEOUT instead of a hang.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>
#include "tv_common.cuh"

namespace tv {
namespace attn {

constexpr int kBM = 128;                       // query rows per M tile
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kNT = 2;                         // M tiles per CTA
constexpr int kStages = 2;                     // K and V ring depth
constexpr int kThreads = 384;                  // 12 warps
constexpr int kPagesPerTile = kBN / kPageSize; // 8
constexpr int kMaxSplits = 16;
constexpr int kMinChunkTiles = 2;              // a split covers at least this many KV tiles
constexpr int kItemsPerCta = 4;                // work items targeted per persistent CTA
constexpr int kRowsPerItem = kNT * kBM;        // partial rows stored per work item
constexpr int kMaxBatch = 4096;
constexpr float kRescaleLog2 = 8.0f;           // lazy O rescale threshold (factor 256)

struct WorkItem {
  int32_t b, g, mp, nt;           // request, KV head, M-tile pair, active M tiles (1 or 2)
  int32_t tile_begin, tile_end;   // KV tiles [begin, end) of 128 keys
  int32_t split, n_splits;        // position among the splits of (b, g, mp)
};

struct Sched {
  int32_t counter;  // next work item (atomic)
  int32_t n_items;
  int32_t pad[62];
};

struct AttnParams {
  CUtensorMap tmQ;
  CUtensorMap tmK;
  CUtensorMap tmV;
  const int32_t* page_table;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint64_t* anc_mask;
  uint16_t* out;       // bf16 bits
  float* lse;
  const WorkItem* items;
  Sched* sched;
  float* part_o;
  float* part_lse;
  int32_t* status;
  int max_pages, n_max, Hq, Hkv, G, q_box_nodes;
  float scale_log2;
};

// shared-memory layout of the main kernel (dynamic part, 1024-byte aligned)
template <int D>
struct Smem {
  static constexpr int kDBlocks = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr int kQTile = kBM * D * 2;
  static constexpr int kKVTile = kBN * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kNT * kQTile;
  static constexpr int kV = kK + kStages * kKVTile;
  static constexpr int kBytes = kV + kStages * kKVTile;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ bool key_visible(int key, int L, int N, uint64_t anc) {
  if (key < L) return true;
  const int j = key - L;
  return j < N && ((anc >> j) & 1ull);
}

// Bounded wait whose outcome is uniform across the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) verify_attn_kernel(const __grid_constant__ AttnParams p) {
  using S = Smem<D>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_kf[kStages], bar_ke[kStages], bar_vf[kStages], bar_ve[kStages];
  __shared__ uint64_t bar_s[kNT], bar_p[kNT], bar_o[kNT];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  __shared__ int item_idx_sh;
  __shared__ WorkItem item_sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_items = p.sched->n_items;
  if (blockIdx.x >= n_items) return;  // fewer items than CTAs

  if (tid == 0) {
    abort_sh = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_kf[s], 1);
      mbar_init(&bar_ke[s], 1);
      mbar_init(&bar_vf[s], 1);
      mbar_init(&bar_ve[s], 1);
    }
    for (int t = 0; t < kNT; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], kBM);
      mbar_init(&bar_o[t], 1);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
  }
  if (warp == 2) {
    tmem_alloc(&tmem_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;

  uint8_t* sQ = smem + S::kQ;
  uint8_t* sK = smem + S::kK;
  uint8_t* sV = smem + S::kV;

  uint32_t kv_it = 0;        // KV tiles consumed so far by this CTA (all roles agree)
  uint32_t items_done = 0;   // work items finished by this CTA
  uint32_t ph_p[kNT] = {0, 0};  // MMA warp: P-ready phases
  uint32_t ph_s = 0;            // softmax warps: S-ready phase of their tile
  uint32_t ph_o = 0;            // softmax warps: O-ready phase of their tile
  int last_b = -1;

  for (;;) {
    if (tid == 0) {
      const int idx = atomicAdd(&p.sched->counter, 1);
      item_idx_sh = idx;
      if (idx < n_items) item_sh = p.items[idx];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int idx = item_idx_sh;
    if (idx >= n_items || abort_sh) break;
    const WorkItem it = item_sh;
    last_b = it.b;
    const int L = p.prefix_len[it.b];
    const int N = p.n_nodes[it.b];
    const int n_tiles = it.tile_end - it.tile_begin;
    const int G = p.G;

    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (elect_one_sync()) {
        const int qrows_per_tile = p.q_box_nodes * G;
        mbar_arrive_expect_tx(&bar_q, (uint32_t)(it.nt * S::kDBlocks * qrows_per_tile * 128));
        const int node0 = it.mp * kNT * (kBM / G);
        for (int t = 0; t < it.nt; ++t)
          for (int db = 0; db < S::kDBlocks; ++db)
            tma_load_4d(sQ + t * S::kQTile + db * (kBM * 128), &p.tmQ, &bar_q, db * 64, it.g * G,
                        node0 + t * (kBM / G), it.b);
        const int32_t* pt = p.page_table + (int64_t)it.b * p.max_pages;
        for (int j = 0; j < n_tiles; ++j) {
          const uint32_t k = kv_it + j;
          const int s = k % kStages;
          const uint32_t ph = (k / kStages) & 1u;
          const int key0 = (it.tile_begin + j) * kBN;
          const int npg = min(kPagesPerTile, (L + N - key0 + kPageSize - 1) / kPageSize);
          const uint32_t bytes = (uint32_t)(npg * kPageSize * D * 2);
          if (!mbar_wait(&bar_ke[s], ph ^ 1u, &abort_sh)) break;
          mbar_arrive_expect_tx(&bar_kf[s], bytes);
          for (int pg = 0; pg < npg; ++pg) {
            const int page = pt[key0 / kPageSize + pg];
            for (int db = 0; db < S::kDBlocks; ++db)
              tma_load_4d(sK + s * S::kKVTile + db * (kBN * 128) + pg * (kPageSize * 128), &p.tmK, &bar_kf[s],
                          db * 64, 0, it.g, page);
          }
          if (!mbar_wait(&bar_ve[s], ph ^ 1u, &abort_sh)) break;
          mbar_arrive_expect_tx(&bar_vf[s], bytes);
          for (int pg = 0; pg < npg; ++pg) {
            const int page = pt[key0 / kPageSize + pg];
            for (int db = 0; db < S::kDBlocks; ++db)
              tma_load_4d(sV + s * S::kKVTile + db * (kBN * 128) + pg * (kPageSize * 128), &p.tmV, &bar_vf[s],
                          db * 64, 0, it.g, page);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (elect_one_sync()) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, false, true);
        auto issue_qk = [&](int t, int s) {
          const uint32_t d = tmem + t * 128;
#pragma unroll
          for (int db = 0; db < S::kDBlocks; ++db)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc_sw128(smem_u32(sQ + t * S::kQTile + db * (kBM * 128) + kk * 32), 16, 1024);
              const uint64_t bd = sdesc_sw128(smem_u32(sK + s * S::kKVTile + db * (kBN * 128) + kk * 32), 16, 1024);
              mma_ss(d, a, bd, idesc_qk, (db | kk) != 0);
            }
        };
        auto issue_pv = [&](int t, int s, bool acc) {
          const uint32_t d = tmem + 256 + t * D;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(smem_u32(sV + s * S::kKVTile + kk * 2048), kBN * 128, 1024);
            mma_ts(d, tmem + t * 128 + kk * 8, bd, idesc_pv, (acc || kk > 0) ? 1u : 0u);
          }
        };
        bool ok = mbar_wait(&bar_q, items_done & 1u, &abort_sh);
        {
          const int s0 = kv_it % kStages;
          ok = ok && mbar_wait(&bar_kf[s0], (kv_it / kStages) & 1u, &abort_sh);
          tc_fence_after();
          if (ok) {
            for (int t = 0; t < it.nt; ++t) {
              issue_qk(t, s0);
              mma_commit(&bar_s[t]);
            }
            mma_commit(&bar_ke[s0]);
          }
        }
        for (int j = 0; j < n_tiles && ok; ++j) {
          const uint32_t k = kv_it + j;
          const int s = k % kStages;
          ok = mbar_wait(&bar_vf[s], (k / kStages) & 1u, &abort_sh);
          const bool has_next = j + 1 < n_tiles;
          const int s1 = (k + 1) % kStages;
          if (ok && has_next) ok = mbar_wait(&bar_kf[s1], ((k + 1) / kStages) & 1u, &abort_sh);
          for (int t = 0; t < it.nt && ok; ++t) {
            ok = mbar_wait(&bar_p[t], ph_p[t], &abort_sh);
            ph_p[t] ^= 1u;
            tc_fence_after();
            if (!ok) break;
            issue_pv(t, s, j > 0);
            if (has_next) {
              issue_qk(t, s1);
              mma_commit(&bar_s[t]);
            } else {
              mma_commit(&bar_o[t]);
            }
          }
          if (!ok) break;
          mma_commit(&bar_ve[s]);
          if (has_next) mma_commit(&bar_ke[s1]);
        }
      }
      __syncwarp();
    } else if (warp >= 4) {
      // ------------------------------------------------------------ softmax + epilogue
      const int t = (warp - 4) >> 2;
      if (t < it.nt) {
        const int r = (warp & 3) * 32 + lane;                 // row of the M tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + t * 128;
        const uint32_t tO = tmem + lane_base + 256 + t * D;
        const int mrow = (it.mp * kNT + t) * kBM + r;
        const int node = mrow / G;
        const int hh = mrow - node * G;
        const bool row_ok = node < N;
        const uint64_t anc = row_ok ? p.anc_mask[(int64_t)it.b * p.n_max + node] : 0ull;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
          ok = warp_wait(&bar_s[t], ph_s, &abort_sh);
          ph_s ^= 1u;
          tc_fence_after();
          if (!ok) break;
          const int key0 = (it.tile_begin + j) * kBN;
          const bool masked = key0 + kBN > L;
          uint32_t v[32];
          // pass 1: row max
          float mx = -INFINITY;
#pragma unroll
          for (int c0 = 0; c0 < kBN; c0 += 32) {
            tmem_ld32(tS + c0, v);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float x = __uint_as_float(v[c]);
              if (masked && !key_visible(key0 + c0 + c, L, N, anc)) x = -INFINITY;
              mx = fmaxf(mx, x);
            }
          }
          const float m_tile = mx * sl2;
          const float m_new = fmaxf(m_run, m_tile);
          const bool grow = m_new > m_run + kRescaleLog2;
          const float alpha = grow ? ex2_approx(m_run - m_new) : 1.f;  // 0 when m_run = -inf
          if (__any_sync(0xffffffffu, grow && j > 0)) {
            // rescale O (PV of the previous tile completed before S of this tile)
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tO + c0, o);
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tmem_st16(tO + c0, o);
              tmem_st16(tO + c0 + 16, o + 16);
            }
          }
          if (grow) {
            l_run *= alpha;
            m_run = m_new;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          // a last tile that runs past the request's data: clear the V rows past it
          if (t == 0 && key0 + kBN > L + N) {
            const int s = (kv_it + j) % kStages;
            const uint32_t vph = ((kv_it + j) / kStages) & 1u;
            ok = warp_wait(&bar_vf[s], vph, &abort_sh);
            if (!ok) break;
            const int vr = L + N - key0;
            uint8_t* vbase = sV + s * S::kKVTile;
            const int nch = (kBN - vr) * 8 * S::kDBlocks;
            for (int q = (warp & 3) * 32 + lane; q < nch; q += kBM) {
              const int db = q % S::kDBlocks;
              const int rest = q / S::kDBlocks;
              const int row = vr + rest / 8;
              *reinterpret_cast<uint4*>(vbase + db * (kBN * 128) + row * 128 + (rest % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
          // pass 2: probabilities -> bf16 P over the S columns already read
          float rs = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < kBN; c0 += 32) {
            tmem_ld32(tS + c0, v);
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0 = __uint_as_float(v[c]) * sl2 - m_use;
              float x1 = __uint_as_float(v[c + 1]) * sl2 - m_use;
              if (masked) {
                if (!key_visible(key0 + c0 + c, L, N, anc)) x0 = -INFINITY;
                if (!key_visible(key0 + c0 + c + 1, L, N, anc)) x1 = -INFINITY;
              }
              const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
              rs += e0 + e1;
              pk[c >> 1] = pack_bf16x2(e0, e1);
            }
            tmem_st16(tS + (c0 >> 1), pk);
          }
          l_run += rs;
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bar_p[t]);
        }
        // epilogue
        if (ok) ok = warp_wait(&bar_o[t], ph_o, &abort_sh);
        ph_o ^= 1u;
        tc_fence_after();
        if (ok) {
          const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
          const float lse_v = l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
          const int h = it.g * G + hh;
          if (it.n_splits == 1) {
            uint16_t* orow = p.out + (((int64_t)it.b * p.n_max + node) * p.Hq + h) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tO + c0, o);
              if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                  pk[c >> 1] = pack_bf16x2(__uint_as_float(o[c]) * inv_l, __uint_as_float(o[c + 1]) * inv_l);
                uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
              }
            }
            if (row_ok && p.lse) p.lse[((int64_t)it.b * p.n_max + node) * p.Hq + h] = lse_v;
          } else {
            const int64_t prow = (int64_t)idx * kRowsPerItem + t * kBM + r;
            float* orow = p.part_o + prow * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tO + c0, o);
              if (row_ok) {
                float4* dst = reinterpret_cast<float4*>(orow + c0);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                       __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
              }
            }
            if (row_ok) p.part_lse[prow] = lse_v;
          }
        }
      }
    }
    kv_it += n_tiles;
    ++items_done;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (abort_sh && tid == 0 && last_b >= 0) atomicOr(p.status + last_b, TV_DEV_TIMEOUT);
  if (warp == 2) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- plan
struct PlanParams {
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const int32_t* page_table;
  int64_t num_pages;
  int max_pages, B, n_max, G, Hkv, target_items, max_items;
  int32_t* status;
  WorkItem* items;
  Sched* sched;
  int32_t* rq_T;      // KV tiles per request (0 when skipped)
  int32_t* rq_MT;     // M tiles per request
  int32_t* rq_items;  // work items per request
  int32_t* rq_order;  // requests by decreasing cost
  int32_t* rq_off;    // first item of each request
};

__device__ __forceinline__ int splits_for(int T, int nt, long long chunk_cost) {
  long long s = ((long long)T * nt + chunk_cost - 1) / chunk_cost;
  const int cap = max(1, min(kMaxSplits, T / kMinChunkTiles));
  return (int)max(1ll, min((long long)cap, s));
}

__global__ void __launch_bounds__(1024) attn_plan_kernel(const PlanParams p) {
  __shared__ unsigned long long s_total;
  __shared__ long long s_chunk;
  __shared__ int s_items;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) s_total = 0;
  __syncthreads();
  // 1. validation (one warp per request) and per-request tile counts
  for (int b = warp; b < p.B; b += 32) {
    const int st = p.status[b];
    const int L = p.prefix_len[b], N = p.n_nodes[b];
    int bits = 0;
    if (st == 0) {
      if (N < 1 || N > p.n_max) {
        bits = TV_DEV_BAD_TREE;
      } else if (L < 0) {
        bits = TV_DEV_CAPACITY;
      } else {
        const long long need = ((long long)L + N + kPageSize - 1) / kPageSize;
        if (need > p.max_pages) {
          bits = TV_DEV_CAPACITY;
        } else {
          bool bad = false;
          for (long long k = lane; k < need; k += 32) {
            const int pg = p.page_table[(int64_t)b * p.max_pages + k];
            bad |= (pg < 0 || (int64_t)pg >= p.num_pages);
          }
          if (__any_sync(0xffffffffu, bad)) bits = TV_DEV_PAGE_OOB;
        }
      }
      if (bits && lane == 0) p.status[b] = st | bits;
    }
    if (lane == 0) {
      const bool ok = st == 0 && bits == 0;
      p.rq_T[b] = ok ? (L + N + kBN - 1) / kBN : 0;
      p.rq_MT[b] = ok ? (N * p.G + kBM - 1) / kBM : 0;
    }
  }
  __syncthreads();
  // 2. total cost in (KV tile x M tile) units
  unsigned long long part = 0;
  for (int b = tid; b < p.B; b += 1024) part += (unsigned long long)p.rq_T[b] * p.rq_MT[b] * p.Hkv;
  atomicAdd(&s_total, part);
  __syncthreads();
  if (tid == 0) {
    const long long tgt = max(1, p.target_items);
    s_chunk = max(1ll, (long long)((s_total + tgt - 1) / tgt));
  }
  __syncthreads();
  const long long chunk = s_chunk;
  // 3. items per request
  for (int b = tid; b < p.B; b += 1024) {
    const int T = p.rq_T[b], MT = p.rq_MT[b];
    int n = 0;
    if (T > 0) {
      const int MP = (MT + kNT - 1) / kNT;
      for (int mp = 0; mp < MP; ++mp) n += splits_for(T, min(kNT, MT - mp * kNT), chunk);
    }
    p.rq_items[b] = n * p.Hkv;
  }
  __syncthreads();
  // 4. order (largest first) and offsets
  if (tid == 0) {
    for (int b = 0; b < p.B; ++b) p.rq_order[b] = b;
    if (p.B <= 256) {
      for (int i = 1; i < p.B; ++i) {
        const int x = p.rq_order[i];
        const long long cx = (long long)p.rq_T[x] * p.rq_MT[x];
        int j = i - 1;
        while (j >= 0 && (long long)p.rq_T[p.rq_order[j]] * p.rq_MT[p.rq_order[j]] < cx) {
          p.rq_order[j + 1] = p.rq_order[j];
          --j;
        }
        p.rq_order[j + 1] = x;
      }
    }
    int off = 0;
    for (int i = 0; i < p.B; ++i) {
      const int b = p.rq_order[i];
      p.rq_off[b] = off;
      off += p.rq_items[b];
    }
    s_items = min(off, p.max_items);
  }
  __syncthreads();
  // 5. write items: one warp per request; (g, mp, split) with split innermost
  for (int b = warp; b < p.B; b += 32) {
    const int T = p.rq_T[b], MT = p.rq_MT[b];
    if (T == 0) continue;
    const int MP = (MT + kNT - 1) / kNT;
    const int nt_last = MT - (MP - 1) * kNT;
    const int s_full = splits_for(T, kNT, chunk);
    const int s_last = splits_for(T, nt_last, chunk);
    const int per_g = (MP - 1) * s_full + s_last;
    const int total = per_g * p.Hkv;
    const int off = p.rq_off[b];
    for (int q = lane; q < total; q += 32) {
      const int g = q / per_g;
      const int rem = q - g * per_g;
      const int mp = min(rem / s_full, MP - 1);
      const int split = rem - mp * s_full;
      const int ns = (mp == MP - 1) ? s_last : s_full;
      WorkItem w;
      w.b = b;
      w.g = g;
      w.mp = mp;
      w.nt = (mp == MP - 1) ? nt_last : kNT;
      w.tile_begin = (int)((long long)split * T / ns);
      w.tile_end = (int)((long long)(split + 1) * T / ns);
      w.split = split;
      w.n_splits = ns;
      if (off + q < p.max_items) p.items[off + q] = w;
    }
  }
  if (tid == 0) {
    p.sched->counter = 0;
    p.sched->n_items = s_items;
  }
}

// ---------------------------------------------------------------- merge
struct MergeParams {
  const WorkItem* items;
  const Sched* sched;
  const float* part_o;
  const float* part_lse;
  const int32_t* n_nodes;
  const int32_t* status;
  uint16_t* out;
  float* lse;
  int max_items, B, n_max, Hq, G;
};

template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const MergeParams p) {
  const int x = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (x < p.max_items) {
    if (x >= p.sched->n_items) return;
    const WorkItem it = p.items[x];
    if (it.n_splits <= 1 || it.split != 0) return;
    if (p.status[it.b] != 0) return;
    const int N = p.n_nodes[it.b];
    const int ns = it.n_splits;
    constexpr int kPer = D / 32;
    for (int r = warp; r < it.nt * kBM; r += 8) {
      const int mrow = it.mp * kRowsPerItem + r;
      const int node = mrow / p.G;
      if (node >= N) continue;
      const int h = it.g * p.G + (mrow - node * p.G);
      float m = -INFINITY;
      for (int s = 0; s < ns; ++s) m = fmaxf(m, p.part_lse[(int64_t)(x + s) * kRowsPerItem + r]);
      float acc[kPer];
#pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
      float wsum = 0.f;
      for (int s = 0; s < ns; ++s) {
        const float ls = p.part_lse[(int64_t)(x + s) * kRowsPerItem + r];
        const float w = (ls == -INFINITY) ? 0.f : __expf(ls - m);
        wsum += w;
        const float* src = p.part_o + ((int64_t)(x + s) * kRowsPerItem + r) * D;
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] += w * src[lane + 32 * c];
      }
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
      uint16_t* dst = p.out + (((int64_t)it.b * p.n_max + node) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < kPer; ++c) {
        const uint32_t pk = pack_bf16x2(acc[c] * inv, 0.f);
        dst[lane + 32 * c] = (uint16_t)(pk & 0xFFFFu);
      }
      if (lane == 0 && p.lse) p.lse[((int64_t)it.b * p.n_max + node) * p.Hq + h] = m + __logf(wsum);
    }
  } else {
    // requests with a non-zero status get zero outputs
    const int b = x - p.max_items;
    if (b >= p.B || p.status[b] == 0) return;
    const int64_t n = (int64_t)p.n_max * p.Hq * D;
    uint16_t* dst = p.out + (int64_t)b * n;
    for (int64_t i = threadIdx.x; i < n; i += 256) dst[i] = 0;
    if (p.lse)
      for (int64_t i = threadIdx.x; i < (int64_t)p.n_max * p.Hq; i += 256) p.lse[(int64_t)b * p.n_max * p.Hq + i] = 0.f;
  }
}

// ---------------------------------------------------------------- host side
struct WsLayout {
  size_t sched, items, part_lse, part_o, rq, total;
  int max_items;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int B, int n_max, int Hq, int Hkv, int D, int num_sms) {
  WsLayout w;
  const int G = Hq / Hkv;
  const int mt_max = (n_max * G + kBM - 1) / kBM;
  const int mp_max = (mt_max + kNT - 1) / kNT;
  const int64_t max_groups = (int64_t)B * Hkv * mp_max;
  const int64_t cap = std::min<int64_t>(max_groups * kMaxSplits, (int64_t)kItemsPerCta * num_sms + max_groups);
  w.max_items = (int)std::max<int64_t>(1, cap);
  w.sched = 0;
  w.items = align256(sizeof(Sched));
  w.part_lse = align256(w.items + sizeof(WorkItem) * (size_t)w.max_items);
  w.part_o = align256(w.part_lse + sizeof(float) * (size_t)w.max_items * kRowsPerItem);
  w.rq = align256(w.part_o + sizeof(float) * (size_t)w.max_items * kRowsPerItem * D);
  w.total = align256(w.rq + sizeof(int32_t) * 5 * (size_t)std::max(B, 1));
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

template <int D>
static int launch_all(AttnParams& ap, const PlanParams& pp, const MergeParams& mp, int num_sms, cudaStream_t st) {
  attn_plan_kernel<<<1, 1024, 0, st>>>(pp);
  TV_CUDA_CHECK(cudaGetLastError());
  TV_CUDA_CHECK(ensure_smem_attr((const void*)verify_attn_kernel<D>, Smem<D>::kAlloc));
  verify_attn_kernel<D><<<num_sms, kThreads, Smem<D>::kAlloc, st>>>(ap);
  TV_CUDA_CHECK(cudaGetLastError());
  attn_merge_kernel<D><<<mp.max_items + mp.B, 256, 0, st>>>(mp);
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
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
  TV_REQUIRE(q && k_cache && v_cache && page_table && prefix_len && n_nodes && anc_mask && out && status,
             TV_ERR_INVALID_ARG, "tv_tree_verify_attn: NULL pointer");
  TV_REQUIRE(page_size == tv::kPageSize, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: page_size %d != 16", page_size);
  TV_REQUIRE(D == 64 || D == 128, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: D = %d not in {64, 128}", D);
  TV_REQUIRE(Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0, TV_ERR_UNSUPPORTED,
             "tv_tree_verify_attn: Hq = %d not a multiple of Hkv = %d", Hq, Hkv);
  const int G = Hq / Hkv;
  TV_REQUIRE(G <= kBM && kBM % G == 0, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: group size %d must divide 128", G);
  TV_REQUIRE(n_max >= 1 && n_max <= tv::kMaxNodes, TV_ERR_UNSUPPORTED,
             "tv_tree_verify_attn: n_max = %d not in [1, 64]", n_max);
  TV_REQUIRE(B >= 0 && B <= kMaxBatch, TV_ERR_UNSUPPORTED, "tv_tree_verify_attn: B = %d not in [0, %d]", B,
             kMaxBatch);
  TV_REQUIRE(num_pages >= 1 && num_pages < (1ll << 31) && max_pages >= 1, TV_ERR_INVALID_ARG,
             "tv_tree_verify_attn: bad page counts");
  TV_REQUIRE(scale > 0.f && std::isfinite(scale), TV_ERR_INVALID_ARG, "tv_tree_verify_attn: scale must be > 0");
  TV_REQUIRE(tv::aligned16(q) && tv::aligned16(k_cache) && tv::aligned16(v_cache) && tv::aligned16(out),
             TV_ERR_INVALID_ARG, "tv_tree_verify_attn: q, caches and out must be 16-byte aligned");
  if (B == 0) return TV_OK;
  const int num_sms = tv::current_sm_count();
  const WsLayout wl = ws_layout(B, n_max, Hq, Hkv, D, num_sms);
  TV_REQUIRE(ws != nullptr && ws_bytes >= wl.total, TV_ERR_WORKSPACE,
             "tv_tree_verify_attn: workspace %zu bytes < %zu", ws_bytes, wl.total);
  TV_REQUIRE(tv::aligned16(ws), TV_ERR_INVALID_ARG, "tv_tree_verify_attn: workspace must be 16-byte aligned");
  uint8_t* wsb = static_cast<uint8_t*>(ws);

  AttnParams ap;
  memset(&ap, 0, sizeof(ap));
  const int q_box_nodes = std::min(kBM / G, n_max);
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)n_max, (uint64_t)B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2, (uint64_t)n_max * Hq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)G, (uint32_t)q_box_nodes, 1};
    TV_REQUIRE(make_map4(&ap.tmQ, q, dims, str, box), TV_ERR_CUDA, "tv_tree_verify_attn: tensor map for q failed");
  }
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)tv::kPageSize, (uint64_t)Hkv, (uint64_t)num_pages};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)tv::kPageSize * D * 2, (uint64_t)Hkv * tv::kPageSize * D * 2};
    const uint32_t box[4] = {64, (uint32_t)tv::kPageSize, 1, 1};
    TV_REQUIRE(make_map4(&ap.tmK, k_cache, dims, str, box) && make_map4(&ap.tmV, v_cache, dims, str, box),
               TV_ERR_CUDA, "tv_tree_verify_attn: tensor map for the KV cache failed");
  }
  Sched* sched = reinterpret_cast<Sched*>(wsb + wl.sched);
  WorkItem* items = reinterpret_cast<WorkItem*>(wsb + wl.items);
  float* part_lse = reinterpret_cast<float*>(wsb + wl.part_lse);
  float* part_o = reinterpret_cast<float*>(wsb + wl.part_o);
  int32_t* rq = reinterpret_cast<int32_t*>(wsb + wl.rq);

  ap.page_table = page_table;
  ap.prefix_len = prefix_len;
  ap.n_nodes = n_nodes;
  ap.anc_mask = anc_mask;
  ap.out = static_cast<uint16_t*>(out);
  ap.lse = lse;
  ap.items = items;
  ap.sched = sched;
  ap.part_o = part_o;
  ap.part_lse = part_lse;
  ap.status = status;
  ap.max_pages = max_pages;
  ap.n_max = n_max;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.G = G;
  ap.q_box_nodes = q_box_nodes;
  ap.scale_log2 = (float)((double)scale * 1.4426950408889634);

  PlanParams pp;
  pp.prefix_len = prefix_len;
  pp.n_nodes = n_nodes;
  pp.page_table = page_table;
  pp.num_pages = num_pages;
  pp.max_pages = max_pages;
  pp.B = B;
  pp.n_max = n_max;
  pp.G = G;
  pp.Hkv = Hkv;
  pp.target_items = kItemsPerCta * num_sms;
  pp.max_items = wl.max_items;
  pp.status = status;
  pp.items = items;
  pp.sched = sched;
  pp.rq_T = rq;
  pp.rq_MT = rq + B;
  pp.rq_items = rq + 2 * B;
  pp.rq_order = rq + 3 * B;
  pp.rq_off = rq + 4 * B;

  MergeParams mp;
  mp.items = items;
  mp.sched = sched;
  mp.part_o = part_o;
  mp.part_lse = part_lse;
  mp.n_nodes = n_nodes;
  mp.status = status;
  mp.out = static_cast<uint16_t*>(out);
  mp.lse = lse;
  mp.max_items = wl.max_items;
  mp.B = B;
  mp.n_max = n_max;
  mp.Hq = Hq;
  mp.G = G;

  cudaStream_t st = tv::as_stream(stream);
  return D == 128 ? launch_all<128>(ap, pp, mp, num_sms, st) : launch_all<64>(ap, pp, mp, num_sms, st);
}
