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
  __shared__ int64_t src_off[kMaxNodes];
  __shared__ int64_t dst_off[kMaxNodes];
  __shared__ int n_moves;
  __shared__ int ok;

  const int per_req = p.n_layers * p.Hkv;
  const int b = blockIdx.x / per_req;
  const int layer = (blockIdx.x % per_req) / p.Hkv;
  const int h = blockIdx.x % p.Hkv;
  const bool leader = (blockIdx.x % per_req) == 0;
  const int L = p.prefix_len[b];
  const int N = p.n_nodes[b];
  const int32_t* path = p.path_nodes + (int64_t)b * p.n_max;
  const int32_t* pt = p.page_table + (int64_t)b * p.max_pages;

  // validation: path shape (thread 0), capacity, page ids of every needed page (all threads)
  const int st = p.status[b];
  const int a_in = p.accept_len[b];
  const int64_t need = ((int64_t)L + N + kPageSize - 1) / kPageSize;
  const bool cap_bad = L < 0 || N < 1 || need > p.max_pages;
  bool oob = false;
  if (st == 0 && !cap_bad)
    for (int64_t pg = threadIdx.x; pg < need; pg += kCommitThreads) oob |= (pt[pg] < 0 || pt[pg] >= p.num_pages);
  oob = __syncthreads_or(oob) != 0;
  if (threadIdx.x == 0) {
    const int a = a_in;
    int bits = 0;
    if (st == 0) {
      if (N < 1 || N > p.n_max || a < 0 || a >= N || path[0] != 0) {
        bits |= TV_DEV_BAD_TREE;
      } else {
        for (int k = 1; k <= a; ++k)
          if (path[k] <= path[k - 1] || path[k] >= N) bits |= TV_DEV_BAD_TREE;
      }
      if (cap_bad) bits |= TV_DEV_CAPACITY;
      else if (oob) bits |= TV_DEV_PAGE_OOB;
      if (bits) atomicOr(p.status + b, bits);
    }
    ok = (st == 0 && bits == 0);
    int m = 0;
    if (ok) {
      for (int k = 1; k <= a; ++k) {
        const int nk = path[k];
        if (nk == k) continue;
        const int s = L + nk, d = L + k;
        src_off[m] = (((int64_t)pt[s / kPageSize] * p.Hkv + h) * kPageSize + s % kPageSize) * D;
        dst_off[m] = (((int64_t)pt[d / kPageSize] * p.Hkv + h) * kPageSize + d % kPageSize) * D;
        ++m;
      }
    }
    n_moves = m;
  }
  __syncthreads();

  if (ok) {
    const int total = n_moves * 2 * kChunksPerRow;
    uint16_t* kl = p.k + (int64_t)layer * p.layer_stride;
    uint16_t* vl = p.v + (int64_t)layer * p.layer_stride;
    uint4 buf[kPerThread];
    // phase 1: read every moved row (K and V) into registers
#pragma unroll
    for (int r = 0; r < kPerThread; ++r) {
      const int c = threadIdx.x + r * kCommitThreads;
      if (c < total) {
        const int mv = c / (2 * kChunksPerRow);
        const int w = c % (2 * kChunksPerRow);
        const uint16_t* base = (w < kChunksPerRow) ? kl : vl;
        buf[r] = *reinterpret_cast<const uint4*>(base + src_off[mv] + (w % kChunksPerRow) * 8);
      }
    }
    __syncthreads();
    // phase 2: write them to their destinations
#pragma unroll
    for (int r = 0; r < kPerThread; ++r) {
      const int c = threadIdx.x + r * kCommitThreads;
      if (c < total) {
        const int mv = c / (2 * kChunksPerRow);
        const int w = c % (2 * kChunksPerRow);
        uint16_t* base = (w < kChunksPerRow) ? kl : vl;
        *reinterpret_cast<uint4*>(base + dst_off[mv] + (w % kChunksPerRow) * 8) = buf[r];
      }
    }
  }

  if (leader) {
    const int a = ok ? p.accept_len[b] : -1;
    for (int k = threadIdx.x; k < p.n_max; k += kCommitThreads) {
      int64_t slot = -1;
      if (k <= a) {
        const int pos = L + k;
        slot = (int64_t)pt[pos / kPageSize] * kPageSize + pos % kPageSize;
      }
      p.slots[(int64_t)b * p.n_max + k] = slot;
    }
    if (threadIdx.x == 0) p.new_len[b] = ok ? L + a + 1 : L;
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
  const int64_t grid = (int64_t)B * n_layers * Hkv;
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
  p.slots = committed_slots;
  p.new_len = new_len;
  p.status = status;
  cudaStream_t s = tv::as_stream(stream);
  if (D == 128)
    tv::kv_commit_kernel<128><<<(unsigned)grid, tv::kCommitThreads, 0, s>>>(p);
  else
    tv::kv_commit_kernel<64><<<(unsigned)grid, tv::kCommitThreads, 0, s>>>(p);
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
