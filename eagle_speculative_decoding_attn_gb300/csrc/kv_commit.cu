// tv_kv_commit_path: keep the accepted branch's K/V, drop the rejected ones.
//
// "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2, sequence
// diagram: after the single verification pass the target stores the KV of
// the accepted branch and discards the wrong branches.  The accepted path
// 0 = n_0 < n_1 < ... < n_a sits at logical positions L + n_k; it is compacted
// to L + k so the cache holds the accepted tokens contiguously after the
// prefix (new length L + a + 1).
//
// Overlap: a destination L + k can be the source L + n_j of an earlier path
// element (n_j = k, j < k).  Each CTA therefore loads every row it moves into
// registers before any store; CTAs touch disjoint (request, layer, head) rows.
#include <algorithm>
#include "tv_common.cuh"

namespace tv {

struct CommitParams {
  uint16_t* k;                  // bf16 bits
  uint16_t* v;
  int64_t layer_stride;         // elements
  int64_t num_pages;
  const int32_t* page_table;
  int max_pages;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const int32_t* accept_len;
  const int32_t* path_nodes;
  int n_max, Hkv, n_layers;
  int ctas_per_req;             // CTAs sharing one request's (layer, head) pairs
  int64_t* slots;
  int32_t* new_len;
  int32_t* status;
};

constexpr int kCommitThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(const CommitParams p) {
  constexpr int kChunksPerRow = D / 8;                 // 16-byte chunks per row
  constexpr int kMaxChunks = (kMaxNodes - 1) * 2 * kChunksPerRow;
  constexpr int kPerThread = (kMaxChunks + kCommitThreads - 1) / kCommitThreads;
  constexpr int kTreePages = (kMaxNodes + kPageSize - 1) / kPageSize + 1;  // pages a tree's positions span
  __shared__ int64_t src_off[kMaxNodes];
  __shared__ int64_t dst_off[kMaxNodes];
  __shared__ int page_sh[kTreePages];
  __shared__ int n_moves_sh, path_bad_sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / p.ctas_per_req;
  const int c_in = blockIdx.x % p.ctas_per_req;  // this CTA takes pairs c_in, c_in + ctas_per_req, ...
  const bool leader = c_in == 0;
  griddep_wait();
  const int L = p.prefix_len[b];
  const int N = p.n_nodes[b];
  const int st = p.status[b];
  const int a = p.accept_len[b];
  const int32_t* path = p.path_nodes + (int64_t)b * p.n_max;
  const int32_t* pt = p.page_table + (int64_t)b * p.max_pages;
  const int64_t need = ((int64_t)L + N + kPageSize - 1) / kPageSize;
  const bool cap_bad = L < 0 || N < 1 || need > p.max_pages;
  const bool shape_ok = N >= 1 && N <= p.n_max && a >= 0 && a < N;
  const int pg0 = L / kPageSize;  // first page of the tree's positions L .. L + N - 1

  bool oob = false;
  if (warp == 0) {
    // the path (entries lane and lane + 32) and the page ids of the tree's positions,
    // all loaded at once; validation and the move list with warp votes
    const bool go = st == 0 && shape_ok;  // the path is checked whatever the capacity
    int nk0 = -1, nk1 = -1, pid = 0;
    if (go) {
      if (lane <= a) nk0 = path[lane];
      if (lane + 32 <= a) nk1 = path[lane + 32];
      if (!cap_bad && lane < kTreePages && pg0 + lane < need) pid = pt[pg0 + lane];
    }
    const int prev0 = __shfl_up_sync(0xffffffffu, nk0, 1);
    const int last0 = __shfl_sync(0xffffffffu, nk0, 31);
    int prev1 = __shfl_up_sync(0xffffffffu, nk1, 1);
    if (lane == 0) prev1 = last0;
    bool bad = false;
    if (go) {
      if (lane == 0) bad |= nk0 != 0;
      else if (lane <= a) bad |= nk0 <= prev0 || nk0 >= N;
      if (lane + 32 <= a) bad |= nk1 <= prev1 || nk1 >= N;
    }
    const bool path_bad = __any_sync(0xffffffffu, bad);
    // moves: path entries k >= 1 with n_k != k, packed in order
    const bool mv0 = go && lane >= 1 && lane <= a && nk0 != lane;
    const bool mv1 = go && lane + 32 <= a && nk1 != lane + 32;
    const unsigned m0 = __ballot_sync(0xffffffffu, mv0), m1 = __ballot_sync(0xffffffffu, mv1);
    const unsigned below = (1u << lane) - 1u;
    // element offset of a position in head 0 (head h adds h * 16 * D)
    auto offs = [&](int pos) {
      const int page = __shfl_sync(0xffffffffu, pid, (pos / kPageSize - pg0) & 31);
      return (((int64_t)page * p.Hkv) * kPageSize + pos % kPageSize) * D;
    };
    const int64_t s0 = offs(L + (mv0 ? nk0 : 0)), d0 = offs(L + (mv0 ? lane : 0));
    const int64_t s1 = offs(L + (mv1 ? nk1 : 0)), d1 = offs(L + (mv1 ? lane + 32 : 0));
    if (!path_bad) {
      if (mv0) {
        const int i = __popc(m0 & below);
        src_off[i] = s0;
        dst_off[i] = d0;
      }
      if (mv1) {
        const int i = __popc(m0) + __popc(m1 & below);
        src_off[i] = s1;
        dst_off[i] = d1;
      }
    }
    if (lane < kTreePages) page_sh[lane] = pid;
    if (lane == 0) {
      n_moves_sh = path_bad ? 0 : __popc(m0) + __popc(m1);
      path_bad_sh = path_bad;
    }
  } else if (st == 0 && !cap_bad) {
    // every page the request needs must be a valid page id
    for (int64_t pg = tid - 32; pg < need; pg += kCommitThreads - 32) oob |= (pt[pg] < 0 || pt[pg] >= p.num_pages);
  }
  oob = __syncthreads_or(oob) != 0;
  int bits = 0;
  if (st == 0) {
    if (!shape_ok || path_bad_sh) bits |= TV_DEV_BAD_TREE;
    if (cap_bad) bits |= TV_DEV_CAPACITY;
    else if (oob) bits |= TV_DEV_PAGE_OOB;
  }
  const bool ok = st == 0 && bits == 0;
  if (tid == 0 && bits) atomicOr(p.status + b, bits);

  if (ok && n_moves_sh > 0) {
    // items (pair, move, chunk) of this CTA's pairs, in batches of whole pairs: a
    // batch reads all its rows into registers, then writes them (a destination can
    // be the source of an earlier move of the same pair, never of another pair)
    const int per_pair = n_moves_sh * 2 * kChunksPerRow;
    const int n_pairs = p.n_layers * p.Hkv;
    const int my_pairs = (n_pairs - c_in + p.ctas_per_req - 1) / p.ctas_per_req;
    const int pairs_per_batch = (kPerThread * kCommitThreads) / per_pair;  // >= 1
    for (int q0 = 0; q0 < my_pairs; q0 += pairs_per_batch) {
      const int items = min(pairs_per_batch, my_pairs - q0) * per_pair;
      uint4 buf[kPerThread];
      auto addr = [&](int f, bool dst) {
        const int pl = f / per_pair, rem = f - pl * per_pair;
        const int pair = c_in + (q0 + pl) * p.ctas_per_req;
        const int layer = pair / p.Hkv, h = pair - layer * p.Hkv;
        const int mv = rem / (2 * kChunksPerRow), w = rem % (2 * kChunksPerRow);
        uint16_t* base = ((w < kChunksPerRow) ? p.k : p.v) + (int64_t)layer * p.layer_stride +
                         (int64_t)h * kPageSize * D;
        return reinterpret_cast<uint4*>(base + (dst ? dst_off[mv] : src_off[mv]) + (w % kChunksPerRow) * 8);
      };
#pragma unroll
      for (int r = 0; r < kPerThread; ++r) {
        const int f = tid + r * kCommitThreads;
        if (f < items) buf[r] = *addr(f, false);
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kPerThread; ++r) {
        const int f = tid + r * kCommitThreads;
        if (f < items) *addr(f, true) = buf[r];
      }
    }
  }

  if (leader) {
    const int acc = ok ? a : -1;
    for (int k = tid; k < p.n_max; k += kCommitThreads) {
      int64_t slot = -1;
      if (k <= acc) {
        const int pos = L + k;
        slot = (int64_t)page_sh[pos / kPageSize - pg0] * kPageSize + pos % kPageSize;
      }
      p.slots[(int64_t)b * p.n_max + k] = slot;
    }
    if (tid == 0) p.new_len[b] = ok ? L + a + 1 : L;
  }
}

}  // namespace tv

extern "C" int tv_kv_commit_path(void* k_cache, void* v_cache, int n_layers, int64_t layer_stride_elems,
                                 int64_t num_pages, const int32_t* page_table, int max_pages,
                                 const int32_t* prefix_len, const int32_t* n_nodes,
                                 const int32_t* accept_len, const int32_t* path_nodes, int B, int n_max,
                                 int Hkv, int D, int page_size, int64_t* committed_slots, int32_t* new_len,
                                 int32_t* status, void* stream) {
  tv::clear_error();
  TV_REQUIRE(k_cache && v_cache && page_table && prefix_len && n_nodes && accept_len && path_nodes &&
                 committed_slots && new_len && status,
             TV_ERR_INVALID_ARG, "tv_kv_commit_path: NULL pointer");
  TV_REQUIRE(page_size == tv::kPageSize, TV_ERR_UNSUPPORTED, "tv_kv_commit_path: page_size %d != 16",
             page_size);
  TV_REQUIRE(D == 64 || D == 128, TV_ERR_UNSUPPORTED, "tv_kv_commit_path: D = %d not in {64, 128}", D);
  TV_REQUIRE(B >= 0 && n_layers >= 1 && Hkv >= 1 && max_pages >= 1 && num_pages >= 1, TV_ERR_INVALID_ARG,
             "tv_kv_commit_path: bad sizes");
  TV_REQUIRE(n_max >= 1 && n_max <= tv::kMaxNodes, TV_ERR_UNSUPPORTED,
             "tv_kv_commit_path: n_max = %d not in [1, 64]", n_max);
  TV_REQUIRE(tv::aligned16(k_cache) && tv::aligned16(v_cache) && layer_stride_elems % 8 == 0,
             TV_ERR_INVALID_ARG, "tv_kv_commit_path: caches and layer stride must be 16-byte aligned");
  TV_REQUIRE(n_layers == 1 || layer_stride_elems >= num_pages * Hkv * tv::kPageSize * (int64_t)D,
             TV_ERR_INVALID_ARG, "tv_kv_commit_path: layer stride smaller than one layer");
  if (B == 0) return TV_OK;
  // a few CTAs per SM in total; each validates its request once and then moves
  // the rows of every ctas_per_req-th (layer, head) pair
  const int64_t pairs = (int64_t)n_layers * Hkv;
  const int64_t want = (4ll * tv::current_sm_count() + B - 1) / B;
  const int ctas_per_req = (int)std::max<int64_t>(1, std::min<int64_t>(pairs, want));
  const int64_t grid = (int64_t)B * ctas_per_req;
  TV_REQUIRE(grid < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_kv_commit_path: grid too large");
  tv::CommitParams p;
  p.k = static_cast<uint16_t*>(k_cache);
  p.v = static_cast<uint16_t*>(v_cache);
  p.layer_stride = layer_stride_elems;
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.prefix_len = prefix_len;
  p.n_nodes = n_nodes;
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.n_max = n_max;
  p.Hkv = Hkv;
  p.n_layers = n_layers;
  p.ctas_per_req = ctas_per_req;
  p.slots = committed_slots;
  p.new_len = new_len;
  p.status = status;
  cudaStream_t s = tv::as_stream(stream);
  if (D == 128)
    TV_CUDA_CHECK(tv::launch_pdl(tv::kv_commit_kernel<128>, dim3((unsigned)grid), dim3(tv::kCommitThreads), 0, s, p));
  else
    TV_CUDA_CHECK(tv::launch_pdl(tv::kv_commit_kernel<64>, dim3((unsigned)grid), dim3(tv::kCommitThreads), 0, s, p));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
