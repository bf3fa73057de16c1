// tv_tree_accept: longest accepted root-to-node path of the draft tree.
//
// Greedy (T = 0): a non-root node hits when its drafted token equals the
// target's argmax at its parent (the argmax rule of "SGLang EAGLE-2
// Speculative Decoding", section 2, applied to the target); the deepest node
// whose whole root path hits is accepted, and the target's argmax there is
// the bonus token (study note "EAGLE", case 1: k hits emit k+1 tokens).
// Sampling (T > 0) runs in tree_accept_sample.cu.
//
// Greedy design: when every node's logits are small enough to read outright,
// one parallel pass reduces every node's row to slice argmaxes and the last
// CTA of a request resolves the walk (greedy_onepass_kernel).  Otherwise a
// level-synchronous walk: one thread-block cluster of CL CTAs per request (8,
// or 4 for a batch whose 8-CTA clusters would not all be resident), CTA r
// owning the vocabulary slice [r*chunk, (r+1)*chunk); rows are read only for
// the frontier nodes, and the per-node argmaxes are combined through
// distributed shared memory in rank order, so every CTA takes identical
// decisions.
#include <cooperative_groups.h>
#include <cfloat>
#include <climits>
#include "tv_common.cuh"
#include "accept_common.cuh"

namespace cg = cooperative_groups;

namespace tv {

constexpr int kCL = 8;             // CTAs per request
constexpr int kMinCL = 4;          // CTAs per request for large batches (all clusters resident)
constexpr int kMaxCL = 8;
constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;

struct AcceptParams {
  const float* target;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* n_nodes;
  int n_max, V, chunk;
  int32_t* accept_len;
  int32_t* path_nodes;
  int32_t* out_tokens;
  int32_t* status;
};

struct __align__(16) ClSlot {
  float f;
  int i;
};

struct AccShared {
  AccTree tr;
  int am[kMaxNodes];
  int front[kMaxNodes];
  int nxt[kMaxNodes];
  int path[kMaxNodes];
  float wf[kAccWarps];
  int wi[kAccWarps];
  ClSlot slot[2];
  ClSlot gath[kMaxCL];  // this exchange's slots of every CTA, copied in (rank order)
  float bf;
  int bi;
  int cnt;
  int lowest;
};

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ void argmax_take(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Block argmax (ties -> lowest index); result in sh.bf / sh.bi.
__device__ void block_argmax(float v, int i, AccShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_take(v, i, v2, i2);
  }
  if (lane == 0) {
    sh.wf[warp] = v;
    sh.wi[warp] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv = sh.wf[0];
    int bi = sh.wi[0];
    for (int w = 1; w < kAccWarps; ++w) argmax_take(bv, bi, sh.wf[w], sh.wi[w]);
    sh.bf = bv;
    sh.bi = bi;
  }
  __syncthreads();
}

// Cluster exchange: thread 0 of every CTA publishes its slot, then every
// thread reads all CL slots in rank order.  Slots are double buffered so a
// slot is never rewritten before every CTA has passed the next cluster barrier.
template <int CL>
struct ClusterEx {
  cg::cluster_group cl;
  int buf;
  __device__ ClusterEx() : cl(cg::this_cluster()), buf(0) {}
  __device__ ClSlot* publish(AccShared& sh) { return &sh.slot[buf]; }
  // cluster barrier, then the first CL threads copy every CTA's slot into this
  // CTA's shared memory (one remote read per slot instead of one per thread)
  __device__ void exchange(AccShared& sh) {
    cl.sync();
    if (threadIdx.x < CL) sh.gath[threadIdx.x] = *cl.map_shared_rank(&sh.slot[buf], (int)threadIdx.x);
    __syncthreads();
  }
  __device__ const ClSlot* got(AccShared& sh, int r) { return &sh.gath[r]; }
  __device__ void sync() { cl.sync(); }
  __device__ void flip() { buf ^= 1; }
};

// ---------------------------------------------------------------- the kernel
template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kAccThreads, 1)
    tree_accept_kernel(const AcceptParams p) {
  __shared__ AccShared sh;
  ClusterEx<CL> ex;
  const int rank = (int)ex.cl.block_rank();
  const int b = blockIdx.x / CL;
  const int tid = threadIdx.x;
  const int n_max = p.n_max, V = p.V;
  const int lo = min(V, rank * p.chunk);
  const int hi = min(V, lo + p.chunk);
  const int len = hi - lo;

  // Everything up to the outputs reads only inputs (tree, tokens, logits) and
  // writes nothing global, so it runs while the previous kernel finishes;
  // status, which that kernel may write, is read and written after the wait
  // before the outputs.  Tree setup and validation: every CTA redundantly,
  // identical results.
  const AccTreeIn tin = acc_tree_load(p.parents, p.tokens, nullptr, nullptr, p.n_nodes, b, n_max);
  const int bad = acc_tree_build(sh.tr, tin, n_max, V);
  int best = 0;
  int bonus = -1;
  if (bad == 0) {  // uniform across the cluster: every CTA computed the same flag
    const bool vec4 = (V & 3) == 0;
    {
      // ================================================ greedy: level-synchronous walk
      int nf = 1;
      if (tid == 0) sh.front[0] = 0;
      __syncthreads();
      while (nf > 0) {
        for (int f = 0; f < nf; ++f) {
          const int node = sh.front[f];
          const float* row = p.target + ((int64_t)b * n_max + node) * V;
          float bv = -FLT_MAX;
          int bi = INT_MAX;
          if (vec4) {
            const float4* r4 = reinterpret_cast<const float4*>(row + lo);
            for (int j = tid; j < (len >> 2); j += kAccThreads) {
              const float4 x = __ldg(r4 + j);
              const int base = lo + 4 * j;
              argmax_take(bv, bi, x.x, base);
              argmax_take(bv, bi, x.y, base + 1);
              argmax_take(bv, bi, x.z, base + 2);
              argmax_take(bv, bi, x.w, base + 3);
            }
          } else {
            for (int j = tid; j < len; j += kAccThreads) argmax_take(bv, bi, __ldg(row + lo + j), lo + j);
          }
          block_argmax(bv, bi, sh);
          if (tid == 0) {
            ClSlot* s = ex.publish(sh);
            s->f = sh.bf;
            s->i = sh.bi;
          }
          ex.exchange(sh);
          float gv = -FLT_MAX;
          int gi = INT_MAX;
          for (int r = 0; r < CL; ++r) {
            const ClSlot* s = ex.got(sh, r);
            argmax_take(gv, gi, s->f, s->i);
          }
          ex.flip();
          if (tid == 0) sh.am[node] = gi;  // identical in every CTA
        }
        __syncthreads();
        if (tid == 0) {
          // next frontier: children of frontier nodes whose token is the parent's argmax
          int cnt = 0, lowest = INT_MAX;
          for (int f = 0; f < nf; ++f) {
            const int node = sh.front[f];
            for (int k = sh.tr.kid_off[node]; k < sh.tr.kid_off[node + 1]; ++k) {
              const int c = sh.tr.kids[k];
              if (sh.tr.tok[c] == sh.am[node]) {
                sh.nxt[cnt++] = c;
                lowest = min(lowest, c);
              }
            }
          }
          for (int k = 0; k < cnt; ++k) sh.front[k] = sh.nxt[k];
          sh.cnt = cnt;
          sh.lowest = lowest;
        }
        __syncthreads();
        nf = sh.cnt;
        if (nf > 0) best = sh.lowest;  // all next-frontier nodes share one depth
        __syncthreads();
      }
      bonus = sh.am[best];
    }
  }  // sh.bad == 0

  // ---- outputs (rank 0), after the previous kernel: a request flagged on entry,
  // or with an invalid tree, gets an empty path
  griddep_wait();
  const int st_in = p.status[b];
  const int bad_out = st_in != 0 ? -1 : bad;
  if (bad_out != 0) {
    if (rank == 0) {
      if (tid == 0) {
        p.accept_len[b] = 0;
        if (bad_out > 0) atomicOr(p.status + b, bad_out);
      }
      for (int k = tid; k < n_max; k += kAccThreads) p.path_nodes[(int64_t)b * n_max + k] = -1;
      for (int k = tid; k <= n_max; k += kAccThreads) p.out_tokens[(int64_t)b * (n_max + 1) + k] = -1;
    }
  } else if (rank == 0 && tid == 0) {
    int len_path = 0;
    for (int j = best; j != 0; j = sh.tr.par[j]) sh.path[len_path++] = j;
    // sh.path holds best .. first child; emit root-first
    int32_t* pn = p.path_nodes + (int64_t)b * n_max;
    int32_t* ot = p.out_tokens + (int64_t)b * (n_max + 1);
    pn[0] = 0;
    for (int k = 1; k <= len_path; ++k) {
      const int nd = sh.path[len_path - k];
      pn[k] = nd;
      ot[k - 1] = sh.tr.tok[nd];
    }
    ot[len_path] = bonus;
    for (int k = len_path + 1; k < n_max; ++k) pn[k] = -1;
    for (int k = len_path + 1; k <= n_max; ++k) ot[k] = -1;
    p.accept_len[b] = len_path;
  }
  ex.sync();  // no CTA exits while others may still read its shared memory
}

// ---------------------------------------------------------------- greedy, one pass
// When the logits of every node are small enough to read outright, the greedy
// walk needs no sequential row reads: CTA (slice, node, request) reduces one
// vocabulary slice of one node's row to a partial argmax, and the last CTA of
// a request to finish (arrival counter) takes every node's argmax and resolves
// the walk in shared memory.  The result is the same deepest fully hit node as
// the level walk above; ancestor sets come from pointer jumping over the
// parent links.
constexpr int kArgThreads = 256;
constexpr int kArgPerThread = 32;                        // floats per thread and slice
constexpr int kArgSlice = kArgThreads * kArgPerThread;   // 8192
constexpr int64_t kOnePassMaxBytes = 64ll << 20;         // logits read by the one-pass walk

struct OnePassParams {
  const float* target;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* n_nodes;
  int n_max, V, n_slices;
  float2* part;        // [B][n_max][n_slices]: (value, index bits) of each slice's argmax
  int32_t* tickets;    // [B] arrivals of this call (zero between calls)
  int32_t* accept_len;
  int32_t* path_nodes;
  int32_t* out_tokens;
  int32_t* status;
};

__device__ void argmax_block256(float& v, int& i, float* wv, int* wi) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_take(v, i, v2, i2);
  }
  if (lane == 0) {
    wv[warp] = v;
    wi[warp] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int w = 1; w < kArgThreads / 32; ++w) argmax_take(v, i, wv[w], wi[w]);
}

__global__ void __launch_bounds__(kArgThreads) greedy_onepass_kernel(const OnePassParams p) {
  __shared__ float wv[kArgThreads / 32];
  __shared__ int wi[kArgThreads / 32];
  __shared__ int last_sh;
  __shared__ int par[kMaxNodes], tok[kMaxNodes], am[kMaxNodes], jmp[kMaxNodes];
  __shared__ unsigned long long anc[kMaxNodes];
  __shared__ unsigned long long hit_sh[2], key_sh[2];
  const int sl = blockIdx.x, node = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int n_max = p.n_max, V = p.V;
  // the slices read only inputs (logits, node counts), so they run while the
  // previous kernel finishes; status, which it may write, is read by the last CTA
  // after the wait below
  const int N = p.n_nodes[b];
  const bool req_ok = N >= 1 && N <= n_max;

  // ---- this slice's partial argmax (lowest index on ties)
  float bv = -FLT_MAX;
  int bi = INT_MAX;
  if (req_ok && node < N) {
    const int lo = sl * kArgSlice;
    const int hi = min(V, lo + kArgSlice);
    const float* row = p.target + ((int64_t)b * n_max + node) * V;
    if ((V & 3) == 0) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      float4 x[kArgPerThread / 4];
#pragma unroll
      for (int u = 0; u < kArgPerThread / 4; ++u) {
        const int j = lo / 4 + u * kArgThreads + tid;
        x[u] = j < hi / 4 ? __ldcs(r4 + j) : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      }
#pragma unroll
      for (int u = 0; u < kArgPerThread / 4; ++u) {
        const int base = 4 * (lo / 4 + u * kArgThreads + tid);
        argmax_take(bv, bi, x[u].x, base);
        argmax_take(bv, bi, x[u].y, base + 1);
        argmax_take(bv, bi, x[u].z, base + 2);
        argmax_take(bv, bi, x[u].w, base + 3);
      }
    } else {
      for (int j = lo + tid; j < hi; j += kArgThreads) argmax_take(bv, bi, __ldcs(row + j), j);
    }
  }
  argmax_block256(bv, bi, wv, wi);
  if (tid == 0) {
    p.part[((int64_t)b * n_max + node) * p.n_slices + sl] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    last_sh = atomicAdd(p.tickets + b, 1) == n_max * p.n_slices - 1;
  }
  __syncthreads();
  if (!last_sh) return;
  griddep_wait();
  __threadfence();

  // ---- the last CTA of request b: validate, then resolve the walk
  int bad = p.status[b] != 0 ? -1 : 0;
  if (!bad && (N < 1 || N > n_max)) bad = TV_DEV_BAD_TREE;
  if (!bad) {
    bool sbad = false, tbad = false;
    if (tid < N) {
      const int pi = p.parents[(int64_t)b * n_max + tid];
      const int ti = p.tokens[(int64_t)b * n_max + tid];
      par[tid] = pi;
      tok[tid] = ti;
      sbad = tid == 0 ? pi != -1 : (pi < 0 || pi >= tid);
      tbad = tid >= 1 && (ti < 0 || ti >= V);
      // this node's argmax over the slices
      const float2* pp = p.part + ((int64_t)b * n_max + tid) * p.n_slices;
      float v = -FLT_MAX;
      int i = INT_MAX;
      for (int s = 0; s < p.n_slices; ++s) {
        const float2 x = __ldcg(pp + s);
        argmax_take(v, i, x.x, __float_as_int(x.y));
      }
      am[tid] = i;
    }
    const int any_s = __syncthreads_or(sbad);
    const int any_t = __syncthreads_or(tbad);
    bad = any_s ? TV_DEV_BAD_TREE : (any_t ? TV_DEV_BAD_TOKEN : 0);
  }
  int32_t* pn = p.path_nodes + (int64_t)b * n_max;
  int32_t* ot = p.out_tokens + (int64_t)b * (n_max + 1);
  if (bad) {
    for (int k = tid; k < n_max; k += kArgThreads) pn[k] = -1;
    for (int k = tid; k <= n_max; k += kArgThreads) ot[k] = -1;
    if (tid == 0) {
      p.accept_len[b] = 0;
      if (bad > 0) atomicOr(p.status + b, bad);
      p.tickets[b] = 0;
    }
    return;
  }
  // ancestor-or-self sets by pointer jumping: after round r a set spans 2^(r+1) links
  if (tid < N) {
    const int pi = tid == 0 ? 0 : par[tid];
    anc[tid] = (1ull << tid) | (1ull << pi);
    jmp[tid] = pi;
  }
  __syncthreads();
#pragma unroll 1
  for (int r = 0; r < 6; ++r) {
    unsigned long long a = 0;
    int j = 0;
    if (tid < N) {
      a = anc[tid] | anc[jmp[tid]];
      j = jmp[jmp[tid]];
    }
    __syncthreads();
    if (tid < N) {
      anc[tid] = a;
      jmp[tid] = j;
    }
    __syncthreads();
  }
  // node i hits iff its token is its parent's argmax; accepted iff every
  // non-root node of its root path hits; the result is the deepest accepted
  // node, lowest index on ties
  const bool hit = tid >= 1 && tid < N && tok[tid] == am[par[tid]];
  const unsigned hb = __ballot_sync(0xffffffffu, hit);
  if (tid < 64 && (tid & 31) == 0) hit_sh[tid >> 5] = hb;
  __syncthreads();
  const unsigned long long hits = hit_sh[0] | (hit_sh[1] << 32) | 1ull;
  unsigned long long key = 0;
  if (tid < N && (anc[tid] & ~hits) == 0)
    key = ((unsigned long long)__popcll(anc[tid]) << 8) | (unsigned long long)(255 - tid);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, key, o);
    key = k2 > key ? k2 : key;
  }
  if (tid < 64 && (tid & 31) == 0) key_sh[tid >> 5] = key;
  __syncthreads();
  const unsigned long long kb = key_sh[0] > key_sh[1] ? key_sh[0] : key_sh[1];
  const int best = 255 - (int)(kb & 255);
  const unsigned long long path = anc[best];
  const int a = __popcll(path) - 1;
  // the k-th set bit of the path set is the k-th node of the path (ancestors sort
  // root-first by index)
  auto path_node = [&](int k) {
    unsigned long long m = path;
    for (int q = 0; q < k; ++q) m &= m - 1;
    return __ffsll((long long)m) - 1;
  };
  for (int k = tid; k < n_max; k += kArgThreads) pn[k] = k <= a ? path_node(k) : -1;
  for (int k = tid; k <= n_max; k += kArgThreads) ot[k] = k < a ? tok[path_node(k + 1)] : (k == a ? am[best] : -1);
  if (tid == 0) {
    p.accept_len[b] = a;
    p.tickets[b] = 0;  // ready for the next call
  }
}

}  // namespace tv

namespace {
// clusters of CL CTAs of the greedy walk resident at once (cached per context);
// -1 when a CUDA call fails
template <int CL>
int active_clusters(int dev) {
  static int known[64] = {};  // per device: clusters of CL that fit at once, plus 1 (0 = not yet known)
  static unsigned long long ctx_of[64] = {};  // the context the count was taken in
  unsigned long long ctx = 0;
  if (tv::current_context_id(&ctx) != cudaSuccess) return -1;
  if (known[dev] == 0 || ctx == 0 || ctx_of[dev] != ctx) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(tv::kAccThreads);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tv::tree_accept_kernel<CL>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    known[dev] = n + 1;
    ctx_of[dev] = ctx;
  }
  return known[dev] - 1;
}

// CTAs per request of the greedy level walk: 8 unless the batch's 8-CTA
// clusters cannot all be resident at once, then 4.  0 when a CUDA call fails.
int accept_cluster_size(int B) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int sms = tv::current_sm_count();
  if ((int64_t)B * tv::kCL <= sms) return tv::kCL;
  const int n8 = active_clusters<tv::kCL>(dev);
  if (n8 < 0) return 0;
  return n8 >= B ? tv::kCL : tv::kMinCL;
}

int onepass_slices(int V) { return (V + tv::kArgSlice - 1) / tv::kArgSlice; }
bool onepass_eligible(int B, int n_max, int V) { return (int64_t)B * n_max * V * 4 <= tv::kOnePassMaxBytes; }
size_t onepass_ws_bytes(int B, int n_max, int V) {
  const size_t part = (size_t)B * n_max * onepass_slices(V) * sizeof(float2);
  return ((part + 255) & ~size_t(255)) + (size_t)B * sizeof(int32_t);
}
}  // namespace

extern "C" size_t tv_tree_accept_workspace(int B, int n_max, int V) {
  if (B <= 0 || n_max <= 0 || V <= 0 || !onepass_eligible(B, n_max, V)) return 0;
  return onepass_ws_bytes(B, n_max, V);
}

extern "C" int tv_tree_accept(const float* target_logits, const float* draft_logits, const int32_t* tokens,
                              const int32_t* parents, const int32_t* n_nodes, const uint64_t* anc_mask,
                              const int32_t* depth, int B, int n_max, int V, float temperature, int flags,
                              const float* u_accept, const float* u_sample, int32_t* accept_len,
                              int32_t* path_nodes, int32_t* out_tokens, void* ws, size_t ws_bytes,
                              int32_t* status, void* stream) {
  (void)anc_mask;
  (void)depth;
  tv::clear_error();
  const bool sampling = temperature > 0.f;
  TV_REQUIRE(target_logits && tokens && parents && n_nodes && accept_len && path_nodes && out_tokens && status,
             TV_ERR_INVALID_ARG, "tv_tree_accept: NULL pointer");
  TV_REQUIRE(!sampling || (draft_logits && u_accept && u_sample), TV_ERR_INVALID_ARG,
             "tv_tree_accept: sampling needs draft_logits, u_accept and u_sample");
  TV_REQUIRE(temperature >= 0.f && temperature == temperature, TV_ERR_INVALID_ARG,
             "tv_tree_accept: temperature must be >= 0");
  TV_REQUIRE((flags & ~TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT) == 0, TV_ERR_INVALID_ARG,
             "tv_tree_accept: unknown flags 0x%x", flags);
  TV_REQUIRE(B >= 0 && V >= 1, TV_ERR_INVALID_ARG, "tv_tree_accept: bad sizes B=%d V=%d", B, V);
  TV_REQUIRE(n_max >= 1 && n_max <= tv::kMaxNodes, TV_ERR_UNSUPPORTED,
             "tv_tree_accept: n_max = %d not in [1, 64]", n_max);
  TV_REQUIRE(tv::aligned16(target_logits) && (!sampling || tv::aligned16(draft_logits)), TV_ERR_INVALID_ARG,
             "tv_tree_accept: logits must be 16-byte aligned");
  if (B == 0) return TV_OK;
  if (sampling)
    return tv::launch_accept_sample(target_logits, draft_logits, tokens, parents, n_nodes, u_accept, u_sample, B,
                                    n_max, V, temperature, (flags & TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT) != 0,
                                    accept_len, path_nodes, out_tokens, status, tv::as_stream(stream));
  if (onepass_eligible(B, n_max, V)) {
    const size_t need = onepass_ws_bytes(B, n_max, V);
    TV_REQUIRE(ws != nullptr && ws_bytes >= need && tv::aligned16(ws), TV_ERR_INVALID_ARG,
               "tv_tree_accept: workspace of %zu bytes (16-byte aligned, zero-filled once) required, got %zu",
               need, ws ? ws_bytes : (size_t)0);
    TV_REQUIRE(B <= 65535, TV_ERR_UNSUPPORTED, "tv_tree_accept: B = %d above 65535", B);
    tv::OnePassParams q;
    q.target = target_logits;
    q.tokens = tokens;
    q.parents = parents;
    q.n_nodes = n_nodes;
    q.n_max = n_max;
    q.V = V;
    q.n_slices = onepass_slices(V);
    q.part = reinterpret_cast<float2*>(ws);
    q.tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + (need - (size_t)B * sizeof(int32_t)));
    q.accept_len = accept_len;
    q.path_nodes = path_nodes;
    q.out_tokens = out_tokens;
    q.status = status;
    TV_CUDA_CHECK(tv::launch_pdl(tv::greedy_onepass_kernel, dim3(q.n_slices, n_max, B), dim3(tv::kArgThreads), 0,
                                 tv::as_stream(stream), q));
    TV_CUDA_CHECK(cudaGetLastError());
    return TV_OK;
  }
  const int cl = accept_cluster_size(B);
  TV_REQUIRE(cl > 0, TV_ERR_CUDA, "tv_tree_accept: cluster occupancy query failed");
  TV_REQUIRE((int64_t)B * cl < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_tree_accept: B too large");
  tv::AcceptParams p;
  p.target = target_logits;
  p.tokens = tokens;
  p.parents = parents;
  p.n_nodes = n_nodes;
  p.n_max = n_max;
  p.V = V;
  p.chunk = ((V + cl - 1) / cl + 3) & ~3;
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.status = status;
  if (cl == tv::kCL)
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kCL>, dim3(B * cl), dim3(tv::kAccThreads), 0,
                                 tv::as_stream(stream), p));
  else
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kMinCL>, dim3(B * cl), dim3(tv::kAccThreads), 0,
                                 tv::as_stream(stream), p));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
