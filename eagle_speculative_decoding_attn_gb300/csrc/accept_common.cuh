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
  float us[kMaxNodes];         // u_sample of each node (sampling)
  unsigned long long cmask[kMaxNodes];  // bit j: node j is a child of node n
};

// One request's tree inputs as thread tid (< n_max) loaded them.
struct AccTreeIn {
  int N, par, tok;
  float ua, us;
};

// Issues the loads of request b's node count and of node tid's parent, token,
// u_accept and u_sample (the uniforms when given); the values are used later
// by acc_tree_build.
__device__ __forceinline__ AccTreeIn acc_tree_load(const int32_t* parents, const int32_t* tokens,
                                                   const float* u_accept, const float* u_sample,
                                                   const int32_t* n_nodes, int b, int n_max) {
  const int tid = threadIdx.x;
  AccTreeIn in{n_nodes[b], -2, 0, 0.f, 0.f};
  if (tid < n_max) {
    in.par = parents[(int64_t)b * n_max + tid];
    in.tok = tokens[(int64_t)b * n_max + tid];
    if (u_accept) in.ua = u_accept[(int64_t)b * n_max + tid];
    if (u_sample) in.us = u_sample[(int64_t)b * n_max + tid];
  }
  return in;
}

// Validates the tree and builds the child lists (ascending child index).
// Every CTA that calls it computes the same result.  Returns 0,
// TV_DEV_BAD_TREE (n_nodes out of [1, n_max], a root that is not -1, a parent
// not below its child) or TV_DEV_BAD_TOKEN (a non-root token outside [0, V)).
// Needs at least 64 threads; ends with a block barrier.
__device__ inline int acc_tree_build(AccTree& t, const AccTreeIn& in, int n_max, int V) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int N = in.N;
  const bool n_ok = N >= 1 && N <= n_max;
  const bool live = n_ok && tid < N;
  const bool sbad = live && (tid == 0 ? in.par != -1 : (in.par < 0 || in.par >= tid));
  const bool tbad = live && tid >= 1 && (in.tok < 0 || in.tok >= V);
  if (tid < kMaxNodes) {
    t.par[tid] = live ? in.par : -2;
    t.tok[tid] = in.tok;
    t.ua[tid] = in.ua;
    t.us[tid] = in.us;
  }
  int bad = 0;
  if (__syncthreads_or(sbad || tbad)) bad = __syncthreads_or(sbad) ? TV_DEV_BAD_TREE : TV_DEV_BAD_TOKEN;
  if (!n_ok) bad = TV_DEV_BAD_TREE;
  if (bad) return bad;  // uniform
  // child masks by ballot: warp w takes nodes w, w + nwarps, ...
  {
    const int p0 = lane >= 1 ? t.par[lane] : -2, p1 = t.par[lane + 32];
    for (int n = warp; n < N; n += nwarps) {
      const unsigned lo = __ballot_sync(0xffffffffu, p0 == n);
      const unsigned hi = __ballot_sync(0xffffffffu, p1 == n);
      if (lane == 0) t.cmask[n] = (unsigned long long)lo | ((unsigned long long)hi << 32);
    }
  }
  __syncthreads();
  if (warp == 0) {
    // offsets: exclusive scan of the child counts, nodes lane and lane + 32
    const int c0 = lane < N ? __popcll(t.cmask[lane]) : 0;
    const int c1 = lane + 32 < N ? __popcll(t.cmask[lane + 32]) : 0;
    int i0 = c0, i1 = c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, i0, o);
      const int y1 = __shfl_up_sync(0xffffffffu, i1, o);
      if (lane >= o) {
        i0 += y0;
        i1 += y1;
      }
    }
    const int tot0 = __shfl_sync(0xffffffffu, i0, 31);
    t.kid_off[lane] = i0 - c0;
    t.kid_off[lane + 32] = tot0 + i1 - c1;
    if (lane == 31) t.kid_off[64] = tot0 + i1;
    __syncwarp();
    // child j goes after its lower-indexed siblings
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      if (j >= 1 && j < N) {
        const int pj = t.par[j];
        t.kids[t.kid_off[pj] + __popcll(t.cmask[pj] & ((1ull << j) - 1ull))] = j;
      }
    }
  }
  __syncthreads();
  return 0;
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
