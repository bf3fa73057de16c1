// tv_tree_build_mask: ancestor bitmask and depth of every draft-tree node.
//
// "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2, "Dynamic
// Tree-Attention Masking": the <= 64-node candidate tree is encoded as
// M in {0,1}^{KxK}, M[i][j] = 1 iff j is an ancestor of i or i itself.  With
// K <= 64 one row of M is one 64-bit word; bit j of anc_mask[b][i] is M[i][j].
#include "tv_common.cuh"

namespace tv {

// One CTA of 64 threads per request; thread i owns node i.
__global__ void __launch_bounds__(64) tree_mask_kernel(const int32_t* __restrict__ parents,
                                                       const int32_t* __restrict__ n_nodes, int n_max,
                                                       uint64_t* __restrict__ anc_mask,
                                                       int32_t* __restrict__ depth,
                                                       int32_t* __restrict__ status) {
  __shared__ int32_t par[kMaxNodes];
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  griddep_wait();
  // a few hundred threads of integer work: the next kernel (the attention, which
  // needs a whole SM per CTA) may start its on-chip prologue beside it
  griddep_launch_dependents();
  const int n = n_nodes[b];
  const bool n_ok = n >= 1 && n <= n_max;
  const int p = i < n_max ? parents[(int64_t)b * n_max + i] : 0;
  par[i] = p;
  bool bad = !n_ok;
  if (n_ok && i < n) bad = (i == 0) ? (p != -1) : (p < 0 || p >= i);
  bad = __syncthreads_or(bad) != 0;

  uint64_t word = 0;
  int d = -1;
  if (!bad && i < n) {
    // parent[j] < j for every j on the way up, so the walk ends at the root
    word = 1ull << i;
    d = 0;
    for (int j = i; j != 0;) {
      j = par[j];
      word |= 1ull << j;
      ++d;
    }
  }
  if (i < n_max) {
    anc_mask[(int64_t)b * n_max + i] = word;
    depth[(int64_t)b * n_max + i] = d;
  }
  if (i == 0) status[b] = bad ? TV_DEV_BAD_TREE : 0;
}

}  // namespace tv

extern "C" int tv_tree_build_mask(const int32_t* parents, const int32_t* n_nodes, int B, int n_max,
                                  uint64_t* anc_mask, int32_t* depth, int32_t* status, void* stream) {
  tv::clear_error();
  TV_REQUIRE(parents && n_nodes && anc_mask && depth && status, TV_ERR_INVALID_ARG,
             "tv_tree_build_mask: NULL pointer");
  TV_REQUIRE(B >= 0, TV_ERR_INVALID_ARG, "tv_tree_build_mask: B = %d < 0", B);
  TV_REQUIRE(n_max >= 1 && n_max <= tv::kMaxNodes, TV_ERR_UNSUPPORTED,
             "tv_tree_build_mask: n_max = %d not in [1, 64]", n_max);
  if (B == 0) return TV_OK;
  TV_CUDA_CHECK(tv::launch_pdl(tv::tree_mask_kernel, dim3(B), dim3(64), 0, tv::as_stream(stream), parents, n_nodes,
                               n_max, anc_mask, depth, status));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
