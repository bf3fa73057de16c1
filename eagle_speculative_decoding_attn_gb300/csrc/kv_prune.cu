// tv_kv_prune_pages: release, without copying, the KV pages that hold only
// rejected tree rows after the accepted path has been committed.
//
// "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), failure mode 2: rejected
// branches leave garbage blocks in the page table; managing the branches as a
// prefix tree frees them at once with no copy.  Section 2's sequence diagram:
// the target keeps the accepted branch's KV and drops the wrong branches.
//
// After the commit request b keeps positions [0, new_len); the page-table
// slots ceil(new_len / 16) .. ceil((L + N) / 16) - 1 hold none of them.  Each
// such slot is cleared to -1 and its physical page's reference count drops by
// one; a page whose count reaches zero is appended to the caller's free list.
// Pages referenced by other sequences (counts above one) stay in use.
//
// One warp per request, one lane per released slot (at most six for a
// 64-node tree); counts change by compare-and-swap so that a count never
// goes below zero.
#include "tv_common.cuh"

namespace tv {

struct PruneParams {
  int32_t* page_table;
  int max_pages;
  int32_t* refcount;
  int64_t num_pages;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const int32_t* new_len;
  int32_t* free_list;
  int64_t free_capacity;
  int32_t* free_count;
  int32_t* status;
};

constexpr uint32_t kCasLimit = 1u << 20;  // retries of one count update (contention is a few lanes)

__global__ void __launch_bounds__(32) kv_prune_kernel(const PruneParams p) {
  const int b = blockIdx.x, lane = threadIdx.x;
  griddep_wait();
  if (p.status[b] != 0) return;
  const int L = p.prefix_len[b], N = p.n_nodes[b], nl = p.new_len[b];
  int bad = 0;
  if (L < 0 || N < 1 || ((int64_t)L + N + kPageSize - 1) / kPageSize > p.max_pages)
    bad = TV_DEV_CAPACITY;
  else if (nl < L + 1 || nl > L + N)
    bad = TV_DEV_BAD_TREE;
  if (bad) {
    if (lane == 0) atomicOr(p.status + b, bad);
    return;
  }
  const int first = (nl + kPageSize - 1) / kPageSize;
  const int last = (L + N + kPageSize - 1) / kPageSize;
  int32_t* row = p.page_table + (int64_t)b * p.max_pages;
  bool oob = false;
  for (int s = first + lane; s < last; s += 32) {
    const int id = row[s];
    oob |= id < 0 || (int64_t)id >= p.num_pages;
  }
  if (__any_sync(0xffffffffu, oob)) {  // nothing is released
    if (lane == 0) atomicOr(p.status + b, TV_DEV_PAGE_OOB);
    return;
  }
  int flags = 0;
  for (int s = first + lane; s < last; s += 32) {
    const int id = row[s];
    row[s] = -1;
    int32_t* cnt = p.refcount + id;
    int cur = *reinterpret_cast<volatile int32_t*>(cnt);
    bool freed = false, done = false;
    for (uint32_t it = 0; it < kCasLimit; ++it) {
      if (cur <= 0) {  // released more often than referenced: the count stays at zero
        flags |= TV_DEV_BAD_REFCOUNT;
        done = true;
        break;
      }
      const int prev = atomicCAS(cnt, cur, cur - 1);
      if (prev == cur) {
        freed = cur == 1;
        done = true;
        break;
      }
      cur = prev;
    }
    if (!done) flags |= TV_DEV_TIMEOUT;
    if (freed) {
      const int slot = atomicAdd(p.free_count, 1);
      if (slot < p.free_capacity)
        p.free_list[slot] = id;
      else
        flags |= TV_DEV_CAPACITY;  // the free list is full: the page is free but not listed
    }
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && flags) atomicOr(p.status + b, flags);
}

}  // namespace tv

extern "C" int tv_kv_prune_pages(int32_t* page_table, int max_pages, int32_t* refcount, int64_t num_pages,
                                 const int32_t* prefix_len, const int32_t* n_nodes, const int32_t* new_len, int B,
                                 int page_size, int32_t* free_list, int64_t free_capacity, int32_t* free_count,
                                 int32_t* status, void* stream) {
  tv::clear_error();
  TV_REQUIRE(page_table && refcount && prefix_len && n_nodes && new_len && free_count && status,
             TV_ERR_INVALID_ARG, "tv_kv_prune_pages: NULL pointer");
  TV_REQUIRE(free_list || free_capacity == 0, TV_ERR_INVALID_ARG,
             "tv_kv_prune_pages: free_list is NULL with free_capacity %lld", (long long)free_capacity);
  TV_REQUIRE(B >= 0 && max_pages >= 1 && num_pages >= 1 && num_pages <= INT32_MAX && free_capacity >= 0,
             TV_ERR_INVALID_ARG, "tv_kv_prune_pages: bad sizes B=%d max_pages=%d num_pages=%lld", B, max_pages,
             (long long)num_pages);
  TV_REQUIRE(page_size == tv::kPageSize, TV_ERR_UNSUPPORTED, "tv_kv_prune_pages: page_size %d (16 supported)",
             page_size);
  if (B == 0) return TV_OK;
  tv::PruneParams p;
  p.page_table = page_table;
  p.max_pages = max_pages;
  p.refcount = refcount;
  p.num_pages = num_pages;
  p.prefix_len = prefix_len;
  p.n_nodes = n_nodes;
  p.new_len = new_len;
  p.free_list = free_list;
  p.free_capacity = free_capacity;
  p.free_count = free_count;
  p.status = status;
  TV_CUDA_CHECK(tv::launch_pdl(tv::kv_prune_kernel, dim3(B), dim3(32), 0, tv::as_stream(stream), p));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
