// Pieces shared by the two tree-verify attention kernels (one CTA per SM, and
// CTA pairs with cta_group::2 MMAs): constants, the kernel parameters, the
// visibility word of the ancestor mask, bounded waits, request checks, and the
// split-KV merge.
#pragma once
#include <cmath>
#include <cstdint>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include "tv_common.cuh"
#include "attn_plan.cuh"

namespace tv {
namespace attn {

constexpr int kBM = 128;                       // query rows per M tile
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kNT = 2;                         // M tiles per work group
constexpr int kStages = 2;                     // K and V ring depth
constexpr int kThreads = 384;                  // 12 warps (bf16 cache)
constexpr int kThreadsQ4 = 640;                // 20 warps (low-bit cache: warps 12-19 decode)
constexpr int kPagesPerTile = kBN / kPageSize; // 8
constexpr int kSoftThreads = 256;              // softmax threads of a CTA (warps 4-11)
constexpr int kRowsPerSlot = kNT * kBM;        // rows of one partial slot
constexpr int kMaxBatch = 1024;
constexpr int kMaxBatchQ4 = 256;               // the 4-bit cache's code ring leaves less room for the plan
constexpr float kRescaleLog2 = 8.0f;           // lazy O rescale threshold (factor 256)
constexpr float kLog2e = 1.4426950408889634f;
// register split: 384 threads x 168 at launch = 128 x 88 (warps 0-3) + 256 x 208 (softmax warps)
constexpr uint32_t kRegsLaunch = 168;
constexpr uint32_t kRegsControl = 88;
constexpr uint32_t kRegsSoftmax = 208;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax == kThreads * kRegsLaunch, "register split must match the launch");
// low-bit cache: 640 threads x 96 at launch = 128 x 80 (warps 0-3) + 256 x 128
// (softmax warps) + 256 x 72 (decoding warps); at 128 registers the softmax reads
// the S row in 64-column halves for its maximum and in 32-column chunks for the
// probabilities
constexpr uint32_t kRegsLaunchQ4 = 96;
constexpr uint32_t kRegsControlQ4 = 80;
constexpr uint32_t kRegsSoftmaxQ4 = 128;
constexpr uint32_t kRegsDecodeQ4 = 72;
static_assert(128 * kRegsControlQ4 + 256 * kRegsSoftmaxQ4 + 256 * kRegsDecodeQ4 == kThreadsQ4 * kRegsLaunchQ4,
              "register split must match the launch");
static_assert(kThreadsQ4 * (kRegsLaunchQ4 + 8) > 65536, "the launch leaves each thread exactly kRegsLaunchQ4");
constexpr int kQ4Group = 32;                   // dims sharing one (scale, zero) pair
constexpr int kHalfKeys = kBN / 2;             // keys of one code slot (half a KV tile)

struct AttnParams {
  const uint16_t* q;    // bf16 bits [B, n_max, Hq, D] (read directly by the CTA-pair kernel)
  CUtensorMap tmQ;
  CUtensorMap tmK;
  CUtensorMap tmV;
  const int32_t* page_table;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint64_t* anc_mask;
  uint16_t* out;        // bf16 bits
  float* lse;
  int32_t* status;
  int32_t* ws_bits;     // [B] device-found status bits of this call (zero between calls)
  int32_t* ws_tickets;  // [B * Hkv * mp_max * 2] split arrival counters (zero between calls)
  int32_t* ws_exit;     // CTA exit counter (zero between calls)
  uint4* part_o;        // [2 * gridDim][D/8][256] 8 x fp16: column group major, rows contiguous
  float* part_lse;      // [2 * gridDim][256] log-sum-exp of each partial row
  float* part_scale;    // [2 * gridDim][256] c of each partial row: its fp16 values are O / c (c = 1, or max |O|)
  // 4-bit cache only: codes [pages][Hkv][16][D/2] bytes, params [pages][Hkv][16][D/16] fp16
  const uint8_t* k_codes;
  const uint8_t* k_params;
  const uint8_t* v_codes;
  const uint8_t* v_params;
  int64_t num_pages;
  int B, max_pages, n_max, Hq, Hkv, G, q_box_nodes, mp_max;
  float scale_log2;
};

// Visibility of the 32 keys [base, base + 32) for a row with ancestor word anc.
__device__ __forceinline__ uint32_t visible32(int base, int L, uint64_t anc) {
  const int off = base - L;  // tree index of the first key
  uint32_t pre, tree;
  if (off >= 0) {
    pre = 0u;
    tree = off < 64 ? (uint32_t)(anc >> off) : 0u;
  } else {
    pre = off <= -32 ? 0xffffffffu : ((1u << (-off)) - 1u);
    tree = -off < 64 ? (uint32_t)(anc << (-off)) : 0u;
  }
  return pre | tree;
}

// Multiplies n columns of this thread's TMEM lane by alpha (the rare lazy
// rescale of an O accumulator; kept out of line so the softmax's hot path
// keeps its registers).
template <int n>
__device__ __noinline__ void rescale_o(uint32_t taddr, float alpha) {
#pragma unroll 1
  for (int c0 = 0; c0 < n; c0 += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + c0, o);
#pragma unroll
    for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
    tmem_st32(taddr + c0, o);
    tmem_st_wait();
  }
}

// Bounded wait whose outcome is uniform across the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Status bits of a request whose shape cannot be processed (it is skipped).
__device__ __forceinline__ int request_shape_bits(int L, int N, int n_max, int max_pages) {
  if (N < 1 || N > n_max) return TV_DEV_BAD_TREE;
  if (L < 0) return TV_DEV_CAPACITY;
  if (((int64_t)L + N + kPageSize - 1) / kPageSize > max_pages) return TV_DEV_CAPACITY;
  return 0;
}


// The last split of a (group, M tile) combines every split's normalised
// partial rows by their log-sum-exp weights: out = sum_s w_s O_s with
// w_s = exp(lse_s - m) / sum_s' exp(lse_s' - m), m = max_s lse_s, and
// lse = m + ln sum_s exp(lse_s - m).  A partial row is stored as fp16 values
// of O_s / c_s with c_s = 1, or c_s = max |O_s| for a row with a value past the
// fp16 range (c_s kept in fp32), so w_s c_s multiplies them.
// The work items are (row, column slice) pairs spread over the kNThr calling
// threads, consecutive threads on consecutive rows so the partial reads
// coalesce; one item loads the log-sum-exps, scales and slices of up to kMB
// splits in a single round trip (kMB * kF 16-byte loads per thread in flight),
// and needs a separate pass for the weights only above kMB splits.
// Rows: query row mrow0 + row of the KV head sits at row prow0 + row of the
// partial slots; slot_of(s) is the partial slot of split s.
template <int D, int kMB, int kF, int kNThr, typename SlotOf>
__device__ void merge_items(const AttnParams& p, const Item& it, int mrow0, int prow0, int n_rows, int r,
                            SlotOf slot_of) {
  constexpr int kSlices = D / (8 * kF);
  const int G = p.G;
  const int ns = it.n_splits;
  const int n_items = n_rows * kSlices;
  for (int w = r; w < n_items; w += kNThr) {
    const int row = w % n_rows;
    const int sl = w / n_rows;
    const int prow = prow0 + row;
    const int mrow = mrow0 + row;
    const int node = mrow / G;
    const int64_t orow_idx = ((int64_t)it.b * p.n_max + node) * p.Hq + it.g * G + (mrow - node * G);
    float m = -INFINITY, wsum = 0.f;
    if (ns > kMB) {
      // maximum and weight sum over every split, batch by batch (online)
      for (int s0 = 0; s0 < ns; s0 += kMB) {
        float ls[kMB];
#pragma unroll
        for (int u = 0; u < kMB; ++u)
          ls[u] = s0 + u < ns ? __ldcg(p.part_lse + (int64_t)slot_of(s0 + u) * kRowsPerSlot + prow) : -INFINITY;
        float mb = m;
#pragma unroll
        for (int u = 0; u < kMB; ++u) mb = fmaxf(mb, ls[u]);
        if (mb == -INFINITY) continue;
        wsum = (m == -INFINITY) ? 0.f : wsum * ex2_approx((m - mb) * kLog2e);
#pragma unroll
        for (int u = 0; u < kMB; ++u) wsum += (ls[u] == -INFINITY) ? 0.f : ex2_approx((ls[u] - mb) * kLog2e);
        m = mb;
      }
    }
    float acc[8 * kF];
#pragma unroll
    for (int c = 0; c < 8 * kF; ++c) acc[c] = 0.f;
    for (int s0 = 0; s0 < ns; s0 += kMB) {
      float ls[kMB], sc[kMB];
      uint4 x[kMB][kF];
#pragma unroll
      for (int u = 0; u < kMB; ++u) {
        if (s0 + u < ns) {
          const int slot = slot_of(s0 + u);
          ls[u] = __ldcg(p.part_lse + (int64_t)slot * kRowsPerSlot + prow);
          sc[u] = __ldcg(p.part_scale + (int64_t)slot * kRowsPerSlot + prow);
          const uint4* src = p.part_o + ((int64_t)slot * (D / 8) + sl * kF) * kRowsPerSlot + prow;
#pragma unroll
          for (int q = 0; q < kF; ++q) x[u][q] = __ldcg(src + q * kRowsPerSlot);
        } else {
          ls[u] = -INFINITY;
          sc[u] = 0.f;
#pragma unroll
          for (int q = 0; q < kF; ++q) x[u][q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (ns <= kMB) {  // one batch: the weights come from the values just loaded
#pragma unroll
        for (int u = 0; u < kMB; ++u) m = fmaxf(m, ls[u]);
#pragma unroll
        for (int u = 0; u < kMB; ++u) wsum += (ls[u] == -INFINITY) ? 0.f : ex2_approx((ls[u] - m) * kLog2e);
      }
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
      for (int u = 0; u < kMB; ++u) {
        const float wv = (ls[u] == -INFINITY) ? 0.f : ex2_approx((ls[u] - m) * kLog2e) * inv * sc[u];
#pragma unroll
        for (int q = 0; q < kF; ++q) {
          const uint32_t hw[4] = {x[u][q].x, x[u][q].y, x[u][q].z, x[u][q].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
            acc[8 * q + 2 * e] += wv * f.x;
            acc[8 * q + 2 * e + 1] += wv * f.y;
          }
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(p.out + orow_idx * D + sl * (8 * kF));
#pragma unroll
    for (int q = 0; q < kF; ++q)
      dst[q] = make_uint4(pack_bf16x2(acc[8 * q], acc[8 * q + 1]), pack_bf16x2(acc[8 * q + 2], acc[8 * q + 3]),
                          pack_bf16x2(acc[8 * q + 4], acc[8 * q + 5]), pack_bf16x2(acc[8 * q + 6], acc[8 * q + 7]));
    if (sl == 0 && p.lse) p.lse[orow_idx] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
  }
}

// A role's first touch of global memory: wait for the previous kernel (its writes
// become visible) and let the next kernel be scheduled; its CTAs take SMs as this
// grid's CTAs exit (an SM running this kernel has no room left for another CTA), and it waits for this grid before reading anything this kernel writes.
__device__ __forceinline__ void after_previous(bool& waited) {
  if (!waited) {
    griddep_wait();
    griddep_launch_dependents();
    waited = true;
  }
}

// Run by every thread of the last CTA to exit, once all CTAs have finished (the
// exit count's acquire, passed on by a barrier, makes their stores visible):
// folds the device-found bits into status and zero-fills each request that is
// skipped or in error (and clears the split tickets after a timeout, since a
// split that gave up never took its ticket).
template <int D>
__device__ void finish_requests(const AttnParams& p, int tid, int nthreads) {
  const int64_t per_req = (int64_t)p.n_max * p.Hq * D;
  bool any_timeout = false;
  for (int b = 0; b < p.B; ++b) {
    const int entry = p.status[b];
    const int bits = __ldcg(p.ws_bits + b) |
                     (entry == 0 ? request_shape_bits(p.prefix_len[b], p.n_nodes[b], p.n_max, p.max_pages) : 0);
    if (entry == 0 && bits == 0) continue;
    any_timeout |= (bits & TV_DEV_TIMEOUT) != 0;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)b * per_req);
    for (int64_t i = tid; i < per_req / 8; i += nthreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse)
      for (int64_t i = tid; i < (int64_t)p.n_max * p.Hq; i += nthreads) p.lse[(int64_t)b * p.n_max * p.Hq + i] = 0.f;
    __syncthreads();
    if (tid == 0) {
      p.status[b] = entry | bits;
      p.ws_bits[b] = 0;
    }
  }
  if (any_timeout) {
    __syncthreads();
    const int64_t n_tick = (int64_t)p.B * p.Hkv * p.mp_max * kNT;
    for (int64_t i = tid; i < n_tick; i += nthreads) p.ws_tickets[i] = 0;
  }
  if (tid == 0) *p.ws_exit = 0;
}

// Launches the CTA-pair kernel (head dim 128, bf16 cache) on up to max_ctas CTAs.
int launch_pair(const AttnParams& ap, int max_ctas, cudaStream_t st);

}  // namespace attn
}  // namespace tv
