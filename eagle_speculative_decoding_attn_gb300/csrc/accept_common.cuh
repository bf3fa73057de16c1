// Pieces shared by the acceptance kernels: the per-request draft tree in shared
// memory (parents, tokens, child lists in ascending index) and its validation.
#pragma once
#include <cstdint>
#include "tv_common.cuh"

namespace tv {

struct AccTree {
  int par[kMaxNodes];
  int tok[kMaxNodes];
  int kid_off[kMaxNodes + 1];  // children of node n: kids[kid_off[n] .. kid_off[n + 1])
  int kids[kMaxNodes];
  float ua[kMaxNodes];         // u_accept of each node (sampling)
  int cnt;
  int bad;
};

// Loads request b's tree (one node per thread), validates it and builds the
// child lists.  Every CTA that calls it computes the same result.  Returns 0,
// TV_DEV_BAD_TREE (n_nodes out of [1, n_max], a root that is not -1, a parent
// not below its child) or TV_DEV_BAD_TOKEN (a non-root token outside [0, V)).
// Needs at least 64 threads; ends with a block barrier.
__device__ inline int acc_tree_setup(AccTree& t, const int32_t* parents, const int32_t* tokens,
                                     const float* u_accept, const int32_t* n_nodes, int b, int n_max, int V) {
  const int tid = threadIdx.x;
  const int N = n_nodes[b];
  const bool n_ok = N >= 1 && N <= n_max;
  bool sbad = false, tbad = false;
  if (n_ok && tid < N) {
    const int pi = parents[(int64_t)b * n_max + tid];
    const int ti = tokens[(int64_t)b * n_max + tid];
    t.par[tid] = pi;
    t.tok[tid] = ti;
    sbad = tid == 0 ? pi != -1 : (pi < 0 || pi >= tid);
    tbad = tid >= 1 && (ti < 0 || ti >= V);
  }
  const bool any_s = __syncthreads_or(sbad) != 0;
  const bool any_t = __syncthreads_or(tbad) != 0;
  const int bad = (!n_ok || any_s) ? TV_DEV_BAD_TREE : (any_t ? TV_DEV_BAD_TOKEN : 0);
  if (bad == 0 && tid < kMaxNodes) {  // warps 0 and 1, whole
    // children of node tid, then the exclusive scan of the counts over the nodes
    int cnt = 0;
    if (tid < N)
      for (int j = 1; j < N; ++j) cnt += t.par[j] == tid;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((tid & 31) >= o) incl += y;
    }
    if (tid == 31) t.cnt = incl;  // warp 0's total
    if (tid < N) {
      t.kid_off[tid] = incl - cnt;
      if (u_accept) t.ua[tid] = u_accept[(int64_t)b * n_max + tid];
    }
  }
  if (tid == 0) t.bad = bad;
  __syncthreads();
  if (bad == 0 && tid < N) {
    if (tid >= 32) t.kid_off[tid] += t.cnt;
    if (tid == N - 1) t.kid_off[N] = N - 1;  // every non-root node is somebody's child
  }
  __syncthreads();
  if (bad == 0 && tid >= 1 && tid < N) {
    // ascending child index within each parent's list
    const int pj = t.par[tid];
    int before = 0;
    for (int k = 1; k < tid; ++k) before += t.par[k] == pj;
    t.kids[t.kid_off[pj] + before] = tid;
  }
  __syncthreads();
  return bad;
}

// Sampling acceptance with every CTA's vocabulary slice in registers
// (tree_accept_sample.cu).  Returns a TV_* code; the error text is set.
int launch_accept_sample(const float* target, const float* draft, const int32_t* tokens, const int32_t* parents,
                         const int32_t* n_nodes, const float* u_accept, const float* u_sample, int B, int n_max,
                         int V, float temperature, bool without_replacement, int32_t* accept_len,
                         int32_t* path_nodes, int32_t* out_tokens, int32_t* status, cudaStream_t stream);

// Largest vocabulary the sampling acceptance holds on chip.
constexpr int kSampleMaxV = 16 * 512 * 32;

}  // namespace tv
